"""Decode-step benchmark of the GB300 attention library.

One STEP is one pass of the decode hot path over one batch of synthetic
input, every layer of the model: for the Whisper workloads [beam reorder of
all layers] then per layer K/V append + causal self-attention + cross-
attention over the 1500 encoder frames; for the Qwen3-ASR workload the fused
GQA step (RMSNorm + NeoX RoPE + append + attention) per layer.  The step is
captured once in a CUDA graph and replayed.

Prints ONE JSON line.  value = tokens/s = sequences per step / step time,
summed over ranks (weak scaling: every rank runs its own batch, no data-path
collective).  Extra keys give the achieved K/V GB/s, the roofline of the
dominant kernel (timed per launch with CUDA events on its stream), the clock
record, an end-to-end figure through host buffers, and the CPU oracle's
throughput on a bounded sample.

  python bench.py [--workload NAME] [--steps K] [--warmup W] [--gpus N]
  python bench.py --impl reference ...   # the CPU oracle as the reference arm
"""
import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from kv_cache_decode_asr_gb300 import synthetic as syn  # noqa: E402

DEFAULT_WORKLOAD = "whisper_large_b32"
WORKLOAD_INDEX = {n: i + 1 for i, n in enumerate(syn.WORKLOADS)}
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024
CSRC = "kv_cache_decode_asr_gb300/csrc/"
DECODE_SOURCES = [CSRC + f for f in ("decode_attn.cu", "decode_attn.cuh", "common.cuh")]
PREFILL_SOURCES = [CSRC + f for f in ("prefill.cu", "tcgen05.cuh", "common.cuh")]


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def load_all_peaks():
    """HBM GB/s and dense bf16 TFLOP/s (burst) with where they came from."""
    hbm, src = load_peaks()
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            tf = float(json.load(f)["bf16_tflops"])
        tsrc = "measured bf16_tflops (burst)"
    except Exception:
        tf, tsrc = 1900.0, "fallback bf16 burst"
    return {"hbm": (hbm, src), "tensor": (tf, tsrc)}


def code_sha(rels):
    """Hash of the code in the given sources with comments and whitespace
    removed, so a comment edit does not orphan a counter record."""
    h = hashlib.sha256()
    for rel in rels:
        with open(os.path.join(ROOT, rel)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        h.update(re.sub(r"\s+", "", src).encode())
    return h.hexdigest()[:16]


TRAFFIC_RECORDS = os.path.join(ROOT, "profiles", "dram_traffic.json")


def recorded_traffic(kernel_sources, workload, kernel):
    """DRAM bytes per launch (dram__bytes_read.sum + dram__bytes_write.sum)
    of one kernel on one workload, from the committed ncu records, if the
    record was taken on the current code of the kernel; else None."""
    try:
        with open(TRAFFIC_RECORDS) as f:
            records = json.load(f)["records"]
    except (OSError, ValueError, KeyError):
        return None
    sha = code_sha(kernel_sources)
    for r in records:
        if r.get("workload") == workload and r.get("kernel") == kernel:
            if r.get("code_sha") != sha:
                return None
            b = r.get("dram_bytes_per_launch")
            return int(b) if isinstance(b, (int, float)) else None
    return None


# --------------------------------------------------------------- clocks ----

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while timing."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        # the raw samples go to a scratch file of this run; the JSON line
        # carries their summary
        self.path = os.path.join(os.environ.get("ASR_BENCH_OUT", tempfile.gettempdir()),
                                 f"asr_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 8:
                    continue
                try:
                    mhz.append(float(parts[0]))
                    mx.append(float(parts[1]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[4:8]):
                    if v.lower() == "active":
                        reasons.add(n)
        loaded = [m for m in mhz if m > 0.5 * (max(mx) if mx else 1)] or mhz
        return {"sm_mhz": statistics.median(loaded) if loaded else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(mhz)}


# ------------------------------------------------------------ workloads ----

class WhisperStep:
    """Whisper decode step: [rearrange] + per layer append, self, cross."""

    def __init__(self, name, cfg, device, rank=0):
        import torch
        from kv_cache_decode_asr_gb300 import ops
        self.name, self.cfg, self.ops = name, cfg, ops
        wi = rank_seed_base(name, rank)
        B, H, hd, Lyr = cfg["B"], cfg["heads"], cfg["head_dim"], cfg["layers"]
        cap, F, beam = cfg["capacity"], cfg["frames"], cfg["beam"]
        self.B, self.H, self.hd, self.L, self.cap, self.F = B, H, hd, Lyr, cap, F
        self.d = d = H * hd
        self.row = 2 * d
        self.G = (B + beam - 1) // beam
        self.beam = beam
        self.rearrange = bool(cfg.get("rearrange"))
        self.scale = hd ** -0.5
        f16 = torch.float16
        # self caches [B][layers][capacity][row]; a second buffer when beams reorder
        self.cache_src = syn.dev_fill_normal_(torch.empty(B, Lyr, cap, self.row, dtype=f16,
                                                          device=device), syn.seed_for(wi, 1))
        self.cache = (torch.empty_like(self.cache_src) if self.rearrange else self.cache_src)
        if self.rearrange:
            self.cache.zero_()
        # cross K/V per layer [layers][G][frames][row]
        self.cross = syn.dev_fill_normal_(torch.empty(Lyr, self.G, F, self.row, dtype=f16,
                                                      device=device), syn.seed_for(wi, 2))
        self.qkv = syn.dev_normal((Lyr, B, 3 * d), syn.seed_for(wi, 3), device)
        self.qx = syn.dev_normal((Lyr, B, d), syn.seed_for(wi, 4), device)
        if cfg["lens"] == "fixed":
            lens = np.full(B, cfg["fixed_len"], np.int32)
        else:
            lens = syn.lens_uniform(B, cfg["len_lo"], cfg["len_hi"], syn.seed_for(wi, 5))
        self.lens_host = lens
        self.lens_src = torch.from_numpy(lens).to(device)
        self.idx_host = (syn.beam_permutation(B, beam, syn.seed_for(wi, 6)) if self.rearrange
                         else np.arange(B, dtype=np.int32))
        self.idx = torch.from_numpy(self.idx_host).to(device)
        self.group_host = syn.beam_groups(B, beam)
        self.group = torch.from_numpy(self.group_host).to(device)
        # the step attends lens_dst keys: the reordered lengths (or the lengths)
        self.lens_eff = lens[self.idx_host] if self.rearrange else lens
        self.lens = torch.from_numpy(self.lens_eff.astype(np.int32)).to(device)
        self.slot = self.lens - 1
        self.out_self = torch.zeros(Lyr, B, d, device=device)
        self.out_cross = torch.zeros(Lyr, B, d, device=device)
        self.ws_self = ops.workspace(ops.OP_SELF_ATTN, B, B, 1, H, hd, device=device)
        self.ws_cross = ops.workspace(ops.OP_CROSS_ATTN, B, self.G, beam, H, hd, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    separate_append = False
    # beam reorder fused into each layer's append + self launch (else one
    # asr_kv_rearrange launch over all layers first)
    separate_reorder = False
    profile_kernel = "cross"

    def fused_reorder(self):
        return self.rearrange and not self.separate_reorder

    # kernels launched by one step
    def launches(self):
        return ((1 if self.rearrange and not self.fused_reorder() else 0) +
                (3 if self.separate_append and not self.fused_reorder() else 2) * self.L)

    def layer_calls(self, l, stream=None):
        ops, d = self.ops, self.d
        cache_l = self.cache[:, l]
        qkv = self.qkv[l]
        if self.fused_reorder():
            self.reorder_self_call(l, stream)
        elif self.separate_append:
            ops.asr_kv_append(qkv[:, d:2 * d], qkv[:, 2 * d:], cache_l, self.slot, self.H,
                              self.hd, self.cap, dev_err=self.err, stream=stream)
            ops.asr_self_attn_step(qkv[:, :d], cache_l, self.lens, self.H, self.hd, self.cap,
                                   self.scale, self.out_self[l], self.ws_self, dev_err=self.err,
                                   stream=stream)
        else:
            # append + self-attention in one launch (same bytes written)
            ops.asr_self_attn_append_step(qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:], cache_l,
                                          self.lens, self.H, self.hd, self.cap, self.scale,
                                          self.out_self[l], self.ws_self, dev_err=self.err,
                                          stream=stream)
        self.cross_call(l, stream)

    def reorder_self_call(self, l, stream=None):
        d, qkv = self.d, self.qkv[l]
        self.ops.asr_self_attn_reorder_append_step(
            qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:], self.cache_src[:, l], self.cache[:, l],
            self.idx, self.lens_src, self.lens, self.H, self.hd, self.cap, self.scale,
            self.out_self[l], self.ws_self, dev_err=self.err, stream=stream)

    def cross_call(self, l, stream=None):
        self.ops.asr_cross_attn_step(self.qx[l], self.cross[l], self.group, self.G, self.beam,
                                     self.H, self.hd, self.F, self.scale, self.out_cross[l],
                                     self.ws_cross, dev_err=self.err, stream=stream)

    def step(self, stream=None):
        if self.rearrange and not self.fused_reorder():
            self.ops.asr_kv_rearrange(self.cache_src, self.cache, self.idx, self.lens_src,
                                      self.lens, self.L, self.row, self.cap,
                                      layer_stride=self.cap * self.row, dev_err=self.err,
                                      stream=stream)
        for l in range(self.L):
            self.layer_calls(l, stream)

    # algorithmic bytes
    def bytes_per_layer(self):
        rb = self.row * 2
        q_out = 2 * self.B * self.d * 4
        self_b = int(self.lens_eff.sum()) * rb + q_out
        cross_b = self.active_groups() * self.F * rb + q_out
        append_b = self.B * rb + self.B * 2 * self.d * 4
        rear_b = 2 * int((self.lens_host[self.idx_host] - 1).sum()) * rb if self.rearrange else 0
        return {"self": self_b, "cross": cross_b, "append": append_b, "rearrange": rear_b}

    def active_groups(self):
        return len(set(self.group_host.tolist()))

    def kv_bytes_per_step(self):
        b = self.bytes_per_layer()
        return self.L * (b["self"] + b["cross"] + b["append"] + b["rearrange"])

    dominant = "cross"
    dominant_kernel = "decode_attn_kernel<64,1> (asr_cross_attn_step)"
    kernel_sources = DECODE_SOURCES

    def dominant_bytes_per_launch(self):
        b = self.bytes_per_layer()
        if self.profile_kernel != "self":
            return b["cross"]
        # the fused reorder also writes the history rows it streams (the
        # standalone reorder's read of them is the self launch's own read)
        return b["self"] + b["append"] + (b["rearrange"] // 2 if self.fused_reorder() else 0)

    def traffic_key(self):
        if self.profile_kernel != "self":
            return "cross"
        return "self+append+reorder" if self.fused_reorder() else "self+append"

    def dominant_call(self, l, stream=None):
        if self.profile_kernel == "self" and self.fused_reorder():
            self.reorder_self_call(l, stream)
        elif self.profile_kernel == "self":
            ops, d = self.ops, self.d
            qkv = self.qkv[l]
            ops.asr_self_attn_append_step(qkv[:, :d], qkv[:, d:2 * d], qkv[:, 2 * d:],
                                          self.cache[:, l], self.lens, self.H, self.hd, self.cap,
                                          self.scale, self.out_self[l], self.ws_self,
                                          dev_err=self.err, stream=stream)
        else:
            self.cross_call(l, stream)

    # per-step inputs and outputs for the end-to-end figure
    def host_io(self):
        import torch
        ins = [self.qkv, self.qx]
        outs = [self.out_self, self.out_cross]
        return ins, outs

    # ---- CPU oracle on a sample: `layers` full layers (all sequences)
    def oracle_layer(self, l, oracle):
        import torch
        cache_l = self.cache[:, l].contiguous() if not self.rearrange else None
        if self.rearrange:
            src = self.cache_src[:, l:l + 1].contiguous()
            src_h = src.view(torch.int16).cpu().numpy().view(np.uint16)
            dst_h = np.zeros_like(src_h)
        else:
            cache_h = cache_l.view(torch.int16).cpu().numpy().view(np.uint16)
        cross_h = self.cross[l].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        qkv = self.qkv[l].cpu().numpy()
        qx = self.qx[l].cpu().numpy()
        d = self.d
        t0 = time.perf_counter()
        if self.rearrange:
            lens_dst, _ = oracle.kv_rearrange(src_h, dst_h, self.idx_host, self.lens_host, self.cap)
            cache_h = np.ascontiguousarray(dst_h[:, 0])
        else:
            lens_dst = self.lens_host
        oracle.kv_append(qkv[:, d:2 * d], qkv[:, 2 * d:], cache_h, lens_dst - 1, self.H, self.hd)
        out_s, _ = oracle.self_attn_step(qkv, cache_h, lens_dst, self.H, self.hd, self.scale,
                                         q_stride=3 * d)
        out_c, _ = oracle.cross_attn_step(qx, cross_h, self.group_host, self.H, self.hd,
                                          self.scale)
        dt = time.perf_counter() - t0
        ref = {"self": out_s, "cross": out_c}
        if self.rearrange:
            # the reordered cache with the appended rows: compared as integers
            # (0 when every f16 bit pattern matches)
            ref["cache_bits"] = cache_h.astype(np.float64)
        return dt, ref

    def gpu_layer_outputs(self, l):
        import torch
        got = {"self": self.out_self[l].cpu().numpy(), "cross": self.out_cross[l].cpu().numpy()}
        if self.rearrange:
            got["cache_bits"] = (self.cache[:, l].contiguous().view(torch.int16).cpu().numpy()
                                 .view(np.uint16).astype(np.float64))
        return got

    def oracle_sample(self, i, oracle):
        """(oracle seconds, fraction of the step, reference, gpu) for layer i."""
        dt, ref = self.oracle_layer(i, oracle)
        return dt, 1.0 / self.L, ref, self.gpu_layer_outputs(i), f"layer {i}"

    def n_samples(self):
        return self.L

    metric = "decode-attn tokens/s (K/V HBM GB/s and fraction of HBM peak alongside)"

    def tokens_per_step(self):
        return self.B

    def roofline(self, launch_ms, peaks):
        peak, src = peaks["hbm"]
        b = self.dominant_bytes_per_launch()
        achieved = b / (launch_ms / 1e3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "bytes_per_launch": b,
                "peak_source": f"{src} hbm_gbs"}


class GqaStep:
    """Qwen3-ASR decode step: the fused GQA step per layer."""

    dominant = "gqa"
    dominant_kernel = "decode_attn_kernel<128,2> (asr_gqa_step)"
    kernel_sources = DECODE_SOURCES

    def __init__(self, name, cfg, device, rank=0):
        import torch
        from kv_cache_decode_asr_gb300 import ops
        self.name, self.cfg, self.ops = name, cfg, ops
        wi = rank_seed_base(name, rank)
        B, Hq, Hkv, hd = cfg["B"], cfg["q_heads"], cfg["kv_heads"], cfg["head_dim"]
        Lyr, cap = cfg["layers"], cfg["capacity"]
        self.B, self.Hq, self.Hkv, self.hd, self.L, self.cap = B, Hq, Hkv, hd, Lyr, cap
        self.row = 2 * Hkv * hd
        self.scale = hd ** -0.5
        self.eps, self.base = cfg["eps"], cfg["rope_base"]
        self.cache = syn.dev_fill_normal_(torch.empty(Lyr, B, cap, self.row, dtype=torch.float16,
                                                      device=device), syn.seed_for(wi, 1))
        self.q = syn.dev_normal((Lyr, B, Hq * hd), syn.seed_for(wi, 2), device)
        self.kn = syn.dev_normal((Lyr, B, Hkv * hd), syn.seed_for(wi, 3), device)
        self.vn = syn.dev_normal((Lyr, B, Hkv * hd), syn.seed_for(wi, 4), device)
        self.wq = syn.dev_normal((Lyr, hd), syn.seed_for(wi, 5), device, mean=cfg["w_mean"],
                                 std=cfg["w_std"])
        self.wk = syn.dev_normal((Lyr, hd), syn.seed_for(wi, 6), device, mean=cfg["w_mean"],
                                 std=cfg["w_std"])
        self.n_past_host = syn.lens_uniform(B, cfg["n_past_lo"], cfg["n_past_hi"],
                                            syn.seed_for(wi, 7))
        self.n_past = torch.from_numpy(self.n_past_host).to(device)
        self.out = torch.zeros(Lyr, B, Hq * hd, device=device)
        self.ws = ops.workspace(ops.OP_GQA_STEP, B, B, 1, Hq, hd, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def launches(self):
        return self.L

    def layer_call(self, l, stream=None):
        self.ops.asr_gqa_step(self.q[l], self.kn[l], self.vn[l], self.wq[l], self.wk[l], self.eps,
                              self.base, self.n_past, self.cache[l], self.cap, self.Hq, self.Hkv,
                              self.hd, self.scale, self.out[l], self.ws, dev_err=self.err,
                              stream=stream)

    def step(self, stream=None):
        for l in range(self.L):
            self.layer_call(l, stream)

    def bytes_per_layer(self):
        rb = self.row * 2
        act = self.B * (2 * self.Hq * self.hd + 2 * self.Hkv * self.hd) * 4
        return {"gqa": int(self.n_past_host.sum()) * rb + self.B * rb + act}

    def kv_bytes_per_step(self):
        return self.L * self.bytes_per_layer()["gqa"]

    def dominant_bytes_per_launch(self):
        return self.bytes_per_layer()["gqa"]

    def traffic_key(self):
        return "gqa"

    def dominant_call(self, l, stream=None):
        self.layer_call(l, stream)

    def host_io(self):
        return [self.q, self.kn, self.vn], [self.out]

    def oracle_layer(self, l, oracle):
        import torch
        cache_h = self.cache[l].contiguous().view(torch.int16).cpu().numpy().view(np.uint16).copy()
        args = [t[l].cpu().numpy() for t in (self.q, self.kn, self.vn, self.wq, self.wk)]
        t0 = time.perf_counter()
        out, _ = oracle.gqa_step(*args, self.eps, self.base, self.n_past_host, cache_h, self.Hq,
                                 self.Hkv, self.hd, self.scale)
        return time.perf_counter() - t0, {"gqa": out}

    def gpu_layer_outputs(self, l):
        return {"gqa": self.out[l].cpu().numpy()}

    def oracle_sample(self, i, oracle):
        dt, ref = self.oracle_layer(i, oracle)
        return dt, 1.0 / self.L, ref, self.gpu_layer_outputs(i), f"layer {i}"

    def n_samples(self):
        return self.L

    metric = WhisperStep.metric

    def tokens_per_step(self):
        return self.B

    roofline = WhisperStep.roofline


class PrefillStep:
    """Qwen3-ASR batched prefill: RMSNorm + RoPE + cache write (a7) and the
    causal tensor-core attention (a8) of B prompts of T tokens, one layer."""

    dominant = "prefill_attention"
    dominant_kernel = "attn_tc_kernel<128,true> (tcgen05, asr_prefill_attention)"
    kernel_sources = PREFILL_SOURCES
    metric = "prefill tokens/s (tensor-core TFLOP/s and fraction of the f16 peak alongside)"

    def __init__(self, name, cfg, device, rank=0):
        import torch
        from kv_cache_decode_asr_gb300 import ops
        self.name, self.cfg, self.ops = name, cfg, ops
        wi = rank_seed_base(name, rank)
        B, T, Hq, Hkv, hd = cfg["B"], cfg["T"], cfg["q_heads"], cfg["kv_heads"], cfg["head_dim"]
        self.B, self.T, self.Hq, self.Hkv, self.hd, self.cap = B, T, Hq, Hkv, hd, cfg["capacity"]
        self.L = 1
        self.row = 2 * Hkv * hd
        self.scale = hd ** -0.5
        self.eps, self.base = cfg["eps"], cfg["rope_base"]
        f16 = torch.float16
        self.q = syn.dev_normal((B, T, Hq * hd), syn.seed_for(wi, 1), device, dtype=f16)
        self.k = syn.dev_normal((B, T, Hkv * hd), syn.seed_for(wi, 2), device, dtype=f16)
        self.v = syn.dev_normal((B, T, Hkv * hd), syn.seed_for(wi, 3), device, dtype=f16)
        self.wq = syn.dev_normal((hd,), syn.seed_for(wi, 4), device, mean=cfg["w_mean"],
                                 std=cfg["w_std"])
        self.wk = syn.dev_normal((hd,), syn.seed_for(wi, 5), device, mean=cfg["w_mean"],
                                 std=cfg["w_std"])
        self.cache = torch.zeros(B, self.cap, self.row, dtype=f16, device=device)
        self.out = torch.zeros(B, T, Hq * hd, device=device)
        self.ws = ops.workspace(ops.OP_PREFILL_ATTN, B, Hkv, 1, Hq, hd, T, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def launches(self):
        return 2

    def step(self, stream=None):
        self.ops.asr_prefill_attn(self.q, self.k, self.v, self.wq, self.wk, self.eps, self.base,
                                  self.Hq, self.Hkv, self.hd, self.scale, self.cache, self.cap,
                                  self.out, self.ws, dev_err=self.err, stream=stream)

    def traffic_key(self):
        return "prefill_attn"

    def dominant_call(self, l, stream=None):
        self.ops.asr_prefill_attention(self.B, self.T, self.Hq, self.Hkv, self.hd, self.scale,
                                       self.cache, self.cap, self.out, self.ws, dev_err=self.err,
                                       stream=stream)

    def flops(self):
        """Causal attention FLOPs: QK^T and PV over the keys at or below each query."""
        return 4 * self.B * self.Hq * self.hd * self.T * (self.T + 1) // 2

    def kv_bytes_per_step(self):
        """Bytes the prefill must move: q, k, v in (f16), cache rows written,
        output written (fp32)."""
        return (self.B * self.T * (self.Hq + 2 * self.Hkv) * self.hd * 2
                + self.B * self.T * self.row * 2 + self.B * self.T * self.Hq * self.hd * 4)

    def tokens_per_step(self):
        return self.B * self.T

    def roofline(self, launch_ms, peaks):
        peak, src = peaks["tensor"]
        f = self.flops()
        achieved = f / (launch_ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "flops_per_launch": f,
                "peak_source": f"{src} (dense f16 taken equal to bf16, the nominal ratio 1:1)"}

    def host_io(self):
        return [self.q, self.k, self.v], [self.out]

    def n_samples(self):
        return self.B

    def oracle_sample(self, i, oracle):
        """The whole prefill of sequence i (all heads and positions)."""
        import torch
        h16 = lambda t: t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        q, k, v = h16(self.q[i:i + 1]), h16(self.k[i:i + 1]), h16(self.v[i:i + 1])
        wq, wk = self.wq.cpu().numpy(), self.wk.cpu().numpy()
        cache = np.zeros((1, self.cap, self.row), np.uint16)
        t0 = time.perf_counter()
        ref, _ = oracle.prefill_attn(q, k, v, wq, wk, self.eps, self.base, self.Hq, self.Hkv,
                                     self.hd, self.scale, cache)
        dt = time.perf_counter() - t0
        return dt, 1.0 / self.B, {"out": ref[0]}, {"out": self.out[i].cpu().numpy()}, \
            f"sequence {i}"


class MhaAttnStep:
    """Large-Whisper multi-head attention of a batch of sequences among
    themselves, one layer: the decoder's prompt prefill (causal, K/V rows
    into the self cache, per-sequence lengths) or the encoder's unmasked
    self-attention over 1500 frames.  One step is one call: a small prep
    (V transposed, cache rows) and the tcgen05 attention."""

    kernel_sources = PREFILL_SOURCES

    def __init__(self, name, cfg, device, rank=0):
        import torch
        from kv_cache_decode_asr_gb300 import ops
        self.name, self.cfg, self.ops = name, cfg, ops
        wi = rank_seed_base(name, rank)
        self.causal = cfg["kind"] == "mha_prefill"
        B, T, H, hd = cfg["B"], cfg["T"], cfg["heads"], cfg["head_dim"]
        self.B, self.T, self.H, self.hd, self.L = B, T, H, hd, 1
        self.scale = hd ** -0.5
        f16 = torch.float16
        self.q = syn.dev_normal((B, T, H * hd), syn.seed_for(wi, 1), device, dtype=f16)
        self.k = syn.dev_normal((B, T, H * hd), syn.seed_for(wi, 2), device, dtype=f16)
        self.v = syn.dev_normal((B, T, H * hd), syn.seed_for(wi, 3), device, dtype=f16)
        if self.causal:
            self.lens_host = syn.lens_uniform(B, cfg["len_lo"], cfg["len_hi"], syn.seed_for(wi, 4))
            self.lens = torch.from_numpy(self.lens_host).to(device)
            self.cap = cfg["capacity"]
            self.cache = torch.zeros(B, self.cap, 2 * H * hd, dtype=f16, device=device)
            op = ops.OP_MHA_PREFILL
        else:
            self.lens_host = np.full(B, T, np.int32)
            self.lens = None
            op = ops.OP_ENCODER_ATTN
        self.out = torch.zeros(B, T, H * hd, device=device)
        self.ws = ops.workspace(op, B, H, 1, H, hd, T, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        kname = f"attn_tc_kernel<{hd},{'true' if self.causal else 'false'}>"
        api = "asr_mha_prefill" if self.causal else "asr_encoder_attn"
        self.dominant = api
        self.dominant_kernel = f"{kname} with its prep kernel ({api}, the whole call)"
        self.metric = ("prompt-prefill tokens/s" if self.causal else "encoder frames/s") + \
            " (tensor-core TFLOP/s and fraction of the f16 peak alongside)"

    def launches(self):
        return 2

    def step(self, stream=None):
        if self.causal:
            self.ops.asr_mha_prefill(self.q, self.k, self.v, self.H, self.hd, self.scale,
                                     self.cache, self.cap, self.out, self.ws, lens=self.lens,
                                     dev_err=self.err, stream=stream)
        else:
            self.ops.asr_encoder_attn(self.q, self.k, self.v, self.H, self.hd, self.scale,
                                      self.out, self.ws, dev_err=self.err, stream=stream)

    def traffic_key(self):
        return self.dominant

    def dominant_call(self, l, stream=None):
        self.step(stream)

    def flops(self):
        """QK^T and PV over the keys each real query attends (causal: j <= t)."""
        L = self.lens_host.astype(np.int64)
        pairs = (L * (L + 1) // 2).sum() if self.causal else (L * L).sum()
        return int(4 * self.H * self.hd * pairs)

    def kv_bytes_per_step(self):
        """q, k, v in (f16, real rows), output out (fp32), cache rows (prefill)."""
        n = int(self.lens_host.sum()) * self.H * self.hd
        return n * 2 * 3 + n * 4 + (n * 2 * 2 if self.causal else 0)

    def tokens_per_step(self):
        return int(self.lens_host.sum())

    def roofline(self, launch_ms, peaks):
        peak, src = peaks["tensor"]
        f = self.flops()
        achieved = f / (launch_ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "flops_per_launch": f,
                "peak_source": f"{src} (dense f16 taken equal to bf16, the nominal ratio 1:1)"}

    def host_io(self):
        return [self.q, self.k, self.v], [self.out]

    def n_samples(self):
        return self.B

    def _h16(self, t):
        import torch
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    def oracle_sample(self, i, oracle):
        """Sequence i, every head and real position."""
        q, k, v = self._h16(self.q[i:i + 1]), self._h16(self.k[i:i + 1]), self._h16(self.v[i:i + 1])
        L = int(self.lens_host[i])
        t0 = time.perf_counter()
        ref, _ = oracle.mha_attn(q, k, v, self.H, self.hd, self.scale, self.causal,
                                 lens=np.array([L], np.int32))
        dt = time.perf_counter() - t0
        got = self.out[i, :L].cpu().numpy()
        return dt, L / self.tokens_per_step(), {"out": ref[0, :L]}, {"out": got}, f"sequence {i}"


class CrossFillStep:
    """The cross K/V of one Large-Whisper decoder layer from the encoder
    output of G utterances: a tcgen05 GEMM (frames x d by d x 2d) with the v
    bias and the f16 pack into the cross cache rows."""

    kernel_sources = [CSRC + f for f in ("cross_fill.cu", "tcgen05.cuh", "common.cuh")]
    dominant = "cross_fill"
    dominant_kernel = "cross_fill_kernel (tcgen05 GEMM + bias + f16 pack, asr_cross_kv_fill)"
    parity_tolerance = 1e-3
    parity_note = "f16 cache rows: error beyond one f16 step of the oracle's value"
    metric = "cross K/V fill: encoder frames/s (tensor-core TFLOP/s and fraction of the f16 peak alongside)"

    def __init__(self, name, cfg, device, rank=0):
        import torch
        from kv_cache_decode_asr_gb300 import ops
        self.name, self.cfg, self.ops = name, cfg, ops
        wi = rank_seed_base(name, rank)
        G, F, d = cfg["G"], cfg["frames"], cfg["d"]
        self.G, self.F, self.d, self.L = G, F, d, 1
        f16 = torch.float16
        self.enc = syn.dev_normal((G, F, d), syn.seed_for(wi, 1), device, dtype=f16)
        self.w = syn.dev_normal((2 * d, d), syn.seed_for(wi, 2), device, std=d ** -0.5, dtype=f16)
        self.bias = syn.dev_normal((d,), syn.seed_for(wi, 3), device)
        self.cross = torch.zeros(G, F, 2 * d, dtype=f16, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)

    def launches(self):
        return 1

    def step(self, stream=None):
        self.ops.asr_cross_kv_fill(self.enc, self.w, self.bias, self.cross, dev_err=self.err,
                                   stream=stream)

    def traffic_key(self):
        return "cross_fill"

    def dominant_call(self, l, stream=None):
        self.step(stream)

    def flops(self):
        return 2 * self.G * self.F * (2 * self.d) * self.d

    def kv_bytes_per_step(self):
        """enc in, W in, cache rows out (f16)."""
        return self.G * self.F * self.d * 2 + 2 * self.d * self.d * 2 + self.G * self.F * 2 * self.d * 2

    def tokens_per_step(self):
        return self.G * self.F

    def roofline(self, launch_ms, peaks):
        peak, src = peaks["tensor"]
        f = self.flops()
        achieved = f / (launch_ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak, "flops_per_launch": f,
                "peak_source": f"{src} (dense f16 taken equal to bf16, the nominal ratio 1:1)"}

    def host_io(self):
        return [self.enc], [self.cross]

    def n_samples(self):
        return self.G

    def _h16(self, t):
        import torch
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    def oracle_sample(self, i, oracle):
        """Utterance i: every frame's K/V row."""
        enc = self._h16(self.enc[i:i + 1])
        w = self._h16(self.w)
        b = self.bias.cpu().numpy()
        ref = np.zeros((1, self.F, 2 * self.d), np.uint16)
        t0 = time.perf_counter()
        oracle.cross_kv_fill(enc, w, b, ref)
        dt = time.perf_counter() - t0
        got = self._h16(self.cross[i:i + 1])
        g = got.view(np.float16).astype(np.float64)
        r = ref.view(np.float16).astype(np.float64)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(r), 2.0 ** -14))) - 10)
        # compared as the excess beyond one f16 step of the reference
        excess = np.maximum(np.abs(g - r) - ulp, 0.0)
        return dt, 1.0 / self.G, {"rows": np.zeros_like(excess)}, {"rows": excess}, f"utterance {i}"


class DecoderStep(WhisperStep):
    """The whole Large-Whisper decoder step around the attention, eight
    launches per layer (kv_cache_decode_asr_gb300.decoder): LayerNorm + qkv,
    append + self-attention, out-projection, LayerNorm + cross query,
    cross-attention, cross out-projection, LayerNorm + fc1 + GELU, fc2.  The
    step starts from its input x (the embedded token, a device copy) and
    ends with the residual stream after the last layer."""

    kernel_sources = DECODE_SOURCES
    dominant = "cross"
    dominant_kernel = "decode_attn_kernel<64,1> (asr_cross_attn_step)"
    profile_kernel = "cross"

    def __init__(self, name, cfg, device, rank=0):
        import torch
        from kv_cache_decode_asr_gb300 import decoder
        super().__init__(name, dict(cfg, lens="uniform", rearrange=False), device, rank)
        self.cfg = cfg
        self.decoder = decoder
        wi = rank_seed_base(name, rank)
        self.inner = cfg["inner"]
        self.p = syn.dev_layer_params(self.L, self.d, self.inner, syn.seed_for(wi, 20), device)
        self.pl = [{k: v[l] for k, v in self.p.items()} for l in range(self.L)]
        self.x_in = syn.dev_normal((self.B, self.d), syn.seed_for(wi, 21), device)
        self.x = self.x_in.clone()
        self.bufs = decoder.DecoderBuffers(self.B, self.d, self.inner, self.H, self.hd, self.G,
                                           self.beam, device)
        self.snaps = None
        self.metric = ("decoder-step tokens/s: the whole Large-Whisper decoder step "
                       "(dense layers + attention; step K/V+weight HBM GB/s alongside)")

    def launches(self):
        return self.decoder.LAUNCHES_PER_LAYER * self.L

    def layer(self, l, stream=None):
        self.decoder.whisper_decoder_layer(self.x, self.pl[l], self.cache[:, l], self.lens,
                                           self.cross[l], self.group, self.F, self.bufs,
                                           dev_err=self.err, stream=stream)

    def step(self, stream=None):
        self.x.copy_(self.x_in)
        for l in range(self.L):
            self.layer(l, stream)

    def weight_bytes_per_layer(self):
        d, inner = self.d, self.inner
        w = (3 * d * d + 3 * d * d + 2 * d * inner) * 2
        b = (3 * d + 3 * d + inner + d + 6 * d) * 4
        return w + b

    def dense_bytes_per_layer(self):
        """The six dense launches of a layer: weights and vectors, activations
        in and out (the residual stream read and written by three of them)."""
        B, d, inner = self.B, self.d, self.inner
        # qkv: x in, qkv out; out: att in, x read + written; cross q: x in, qx
        # out; cross out: attc in, x read + written; fc1: x in, h out; fc2: h
        # in, x read + written
        act = 4 * B * ((d + 3 * d) + (d + 2 * d) + (d + d) + (d + 2 * d) + (d + inner) +
                       (inner + 2 * d))
        return self.weight_bytes_per_layer() + act

    def kv_bytes_per_step(self):
        """K/V read and written by the attention plus the dense layers' bytes."""
        return super().kv_bytes_per_step() + self.L * self.dense_bytes_per_layer()

    def extra_rooflines(self, stream, peaks):
        """The dense launches alone (six per layer, every layer, one graph):
        algorithmic bytes per layer / time per layer, against HBM."""
        import torch
        ops = self.ops
        g = torch.cuda.CUDAGraph()
        bufs, x = self.bufs, self.x
        wl = bufs.ws_lin
        with torch.cuda.graph(g, stream=stream):
            for l in range(self.L):
                p = self.pl[l]
                ops.asr_linear(x, p["w_qkv"], bufs.qkv, bias=p["b_qkv"],
                               ln=(p["ln1_g"], p["ln1_b"]), ws=wl, dev_err=self.err)
                ops.asr_linear(bufs.att, p["w_o"], x, bias=p["b_o"], mode="residual", ws=wl,
                               dev_err=self.err)
                ops.asr_linear(x, p["w_cq"], bufs.qx, bias=p["b_cq"],
                               ln=(p["ln2_g"], p["ln2_b"]), ws=wl, dev_err=self.err)
                ops.asr_linear(bufs.attc, p["w_co"], x, bias=p["b_co"], mode="residual", ws=wl,
                               dev_err=self.err)
                ops.asr_linear(x, p["w_fc1"], bufs.h, bias=p["b_fc1"],
                               ln=(p["ln3_g"], p["ln3_b"]), mode="gelu", ws=wl, dev_err=self.err)
                ops.asr_linear(bufs.h, p["w_fc2"], x, bias=p["b_fc2"], mode="residual", ws=wl,
                               dev_err=self.err)
        reps = 20
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        layer_ms = e0.elapsed_time(e1) / (reps * self.L)
        peak, src = peaks["hbm"]
        b = self.dense_bytes_per_layer()
        achieved = b / (layer_ms / 1e3) / 1e9
        return {"roofline_dense": {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "bytes_per_layer": b, "launches_per_layer": 6,
            "us_per_layer": layer_ms * 1e3, "us_per_launch": layer_ms * 1e3 / 6,
            "kernel": "linear_kernel (asr_linear: LayerNorm + tcgen05 product + epilogue)",
            "traffic": None, "peak_source": f"{src} hbm_gbs"}}

    def host_io(self):
        return [self.x_in], [self.x]

    # ---- CPU oracle: whole layers, from the GPU's own input to each layer
    def _host_layer(self, l):
        import torch
        out = {}
        for k, v in self.pl[l].items():
            if v.dtype == torch.float16:
                out[k] = v.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            else:
                out[k] = v.contiguous().cpu().numpy()
        return out

    def _snapshots(self):
        import torch
        if self.snaps is None:
            torch.cuda.synchronize()
            self.x.copy_(self.x_in)
            snaps = [self.x.clone()]
            for l in range(self.L):
                self.layer(l)
                snaps.append(self.x.clone())
            torch.cuda.synchronize()
            self.snaps = [t.cpu().numpy() for t in snaps]
        return self.snaps

    def oracle_sample(self, i, oracle):
        """Layer i of every sequence, from the GPU's input to that layer."""
        import torch
        snaps = self._snapshots()
        p = self._host_layer(i)
        cache = self.cache[:, i].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        cross = self.cross[i].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        t0 = time.perf_counter()
        ref, _ = oracle.whisper_decoder_layer_step(snaps[i], p, cache, self.lens_eff, cross,
                                                   self.group_host, self.H, self.hd)
        dt = time.perf_counter() - t0
        return dt, 1.0 / self.L, {"x": ref}, {"x": snaps[i + 1]}, f"layer {i}"


class QwenDecoderStep(GqaStep):
    """The whole Qwen3-ASR decoder step around the GQA step, five launches
    per layer (kv_cache_decode_asr_gb300.decoder.qwen3_decoder_layer):
    RMSNorm + q/k/v, the fused GQA step, the output projection, RMSNorm +
    gate/up, SwiGLU + down.  The step starts from its input x (the embedded
    token, a device copy) and ends with the residual stream after the last
    layer."""

    dominant = "gqa"
    dominant_kernel = "decode_attn_kernel<128,2> (asr_gqa_step)"

    def __init__(self, name, cfg, device, rank=0):
        from kv_cache_decode_asr_gb300 import decoder
        super().__init__(name, cfg, device, rank)
        self.decoder = decoder
        wi = rank_seed_base(name, rank)
        self.d, self.inner = cfg["d"], cfg["inner"]
        self.p = syn.dev_qwen_layer_params(self.L, self.d, self.inner, self.Hq, self.Hkv, self.hd,
                                           syn.seed_for(wi, 20), device)
        self.pl = [{k: v[l] for k, v in self.p.items()} for l in range(self.L)]
        self.x_in = syn.dev_normal((self.B, self.d), syn.seed_for(wi, 21), device)
        self.x = self.x_in.clone()
        self.bufs = decoder.QwenDecoderBuffers(self.B, self.d, self.inner, self.Hq, self.Hkv,
                                               self.hd, device)
        self.snaps = None
        self.metric = ("decoder-step tokens/s: the whole Qwen3-ASR decoder step "
                       "(dense layers + GQA step; step K/V+weight HBM GB/s alongside)")

    def launches(self):
        return self.decoder.QWEN_LAUNCHES_PER_LAYER * self.L

    def layer(self, l, stream=None):
        self.decoder.qwen3_decoder_layer(self.x, self.pl[l], self.cache[l], self.n_past, self.bufs,
                                         eps=self.eps, rope_base=self.base, dev_err=self.err,
                                         stream=stream)

    def step(self, stream=None):
        self.x.copy_(self.x_in)
        for l in range(self.L):
            self.layer(l, stream)

    def dense_bytes_per_layer(self):
        """The four dense launches of a layer: weights, norm vectors, and the
        activations read and written."""
        B, d, I, nq, nk = self.B, self.d, self.inner, self.Hq * self.hd, self.Hkv * self.hd
        w = 2 * ((nq + 2 * nk) * d + d * nq + 2 * I * d + d * I) + 4 * 2 * d
        act = 4 * B * ((d + nq + 2 * nk) + (nq + 2 * d) + (d + 2 * I) + (2 * I + 2 * d))
        return w + act

    def kv_bytes_per_step(self):
        return super().kv_bytes_per_step() + self.L * self.dense_bytes_per_layer()

    def extra_rooflines(self, stream, peaks):
        import torch
        ops, bufs, x = self.ops, self.bufs, self.x
        wl = bufs.ws_lin
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            for l in range(self.L):
                p = self.pl[l]
                ops.asr_linear(x, p["w_qkv"], bufs.qkv, rms=p["rms1"], eps=self.eps, ws=wl,
                               dev_err=self.err)
                ops.asr_linear(bufs.att, p["w_o"], x, mode="residual", ws=wl, dev_err=self.err)
                ops.asr_linear(x, p["w_gu"], bufs.gu, rms=p["rms2"], eps=self.eps, ws=wl,
                               dev_err=self.err)
                ops.asr_linear(bufs.gu, p["w_down"], x, swiglu=True, mode="residual", ws=wl,
                               dev_err=self.err)
        reps = 20
        with torch.cuda.stream(stream):
            for _ in range(3):
                g.replay()
            e0 = torch.cuda.Event(enable_timing=True)
            e1 = torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        e1.synchronize()
        layer_ms = e0.elapsed_time(e1) / (reps * self.L)
        peak, src = peaks["hbm"]
        b = self.dense_bytes_per_layer()
        achieved = b / (layer_ms / 1e3) / 1e9
        return {"roofline_dense": {
            "bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "bytes_per_layer": b, "launches_per_layer": 4,
            "us_per_layer": layer_ms * 1e3, "us_per_launch": layer_ms * 1e3 / 4,
            "kernel": "linear_kernel (asr_linear: RMSNorm / SwiGLU + tcgen05 product)",
            "traffic": None, "peak_source": f"{src} hbm_gbs"}}

    def host_io(self):
        return [self.x_in], [self.x]

    def _host_layer(self, l):
        import torch
        out = {}
        for k, v in self.pl[l].items():
            if v.dtype == torch.float16:
                out[k] = v.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
            else:
                out[k] = v.contiguous().cpu().numpy()
        return out

    def _snapshots(self):
        import torch
        if self.snaps is None:
            torch.cuda.synchronize()
            self.x.copy_(self.x_in)
            snaps = [self.x.clone()]
            for l in range(self.L):
                self.layer(l)
                snaps.append(self.x.clone())
            torch.cuda.synchronize()
            self.snaps = [t.cpu().numpy() for t in snaps]
        return self.snaps

    def oracle_sample(self, i, oracle):
        """Layer i of every sequence, from the GPU's input to that layer."""
        import torch
        snaps = self._snapshots()
        p = self._host_layer(i)
        cache = self.cache[i].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
        t0 = time.perf_counter()
        ref, _ = oracle.qwen3_decoder_layer_step(snaps[i], p, cache, self.n_past_host, self.Hq,
                                                 self.Hkv, self.hd, eps=self.eps,
                                                 rope_base=self.base)
        dt = time.perf_counter() - t0
        return dt, 1.0 / self.L, {"x": ref}, {"x": snaps[i + 1]}, f"layer {i}"


def make_workload(name, device, rank=0, layers=0):
    cfg = dict(syn.WORKLOADS[name])
    if layers:
        cfg["layers"] = layers
    if cfg["kind"] == "whisper":
        return WhisperStep(name, cfg, device, rank)
    if cfg["kind"] == "gqa":
        return GqaStep(name, cfg, device, rank)
    if cfg["kind"] == "prefill":
        return PrefillStep(name, cfg, device, rank)
    if cfg["kind"] in ("mha_prefill", "encoder"):
        return MhaAttnStep(name, cfg, device, rank)
    if cfg["kind"] == "cross_fill":
        return CrossFillStep(name, cfg, device, rank)
    if cfg["kind"] == "decoder_step":
        return DecoderStep(name, cfg, device, rank)
    if cfg["kind"] == "qwen_decoder_step":
        return QwenDecoderStep(name, cfg, device, rank)
    raise SystemExit(f"workload {name}: not a decode-step bench line")


# ------------------------------------------------------------ helpers -----

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def max_over_ranks(x, world, device):
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_seed_base(name, rank):
    """Seed base of one rank's synthetic batch.  Weak scaling shards nothing:
    every rank draws its own batch of the workload's full per-GPU size from
    seeds no other rank uses (ranks 100 apart, workloads 1 apart)."""
    return WORKLOAD_INDEX[name] + 100 * rank


def job_throughput(ms_total_rank, steps, tokens_per_rank_step, world, device):
    """The slowest rank's timed region sets the step time; the job's value is
    the tokens all ranks processed per second of it."""
    ms_total = max_over_ranks(ms_total_rank, world, device)
    ms_step = ms_total / steps
    return ms_step, tokens_per_rank_step * world / (ms_step / 1e3)


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def cpu_count():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


# ------------------------------------------------------------- our arm ----

# The five decode/prefill configurations the headline metric is stated for;
# the default run measures each of them in the same process (``configs``).
CONFIG_WORKLOADS = ["whisper_tiny_b1", "whisper_tiny_b64_beam5", "whisper_large_b32",
                    "qwen3_asr_gqa_b16", "qwen3_asr_prefill_b8"]


def capture_step(wl, stream):
    """Run the step twice, then capture it in one CUDA graph."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(2):
            wl.step()
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        wl.step()
    torch.cuda.synchronize()
    if int(wl.err.item()) != 0:
        raise RuntimeError(f"{wl.name}: device error flags {int(wl.err.item()):#x}")
    return graph


def time_graph(graph, stream, steps, warmup, world=1):
    """Milliseconds of `steps` back-to-back replays (CUDA events on the
    launching stream, barrier and synchronisation on both sides)."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            graph.replay()
    stream.synchronize()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(steps):
            graph.replay()
        ev1.record(stream)
    ev1.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1)


def time_dominant(wl, stream):
    """The dominant kernel: a CUDA graph of back-to-back launches of it, one
    per layer (each on its own layer's data, together larger than L2), timed
    with CUDA events on the launching stream; milliseconds per launch."""
    import torch
    dom_graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(dom_graph, stream=stream):
        for l in range(wl.L):
            wl.dominant_call(l)
    reps = max(3, min(200, 2000 // max(wl.L, 1)))
    with torch.cuda.stream(stream):
        for _ in range(3):
            dom_graph.replay()
        d0 = torch.cuda.Event(enable_timing=True)
        d1 = torch.cuda.Event(enable_timing=True)
        d0.record(stream)
        for _ in range(reps):
            dom_graph.replay()
        d1.record(stream)
    d1.synchronize()
    return d0.elapsed_time(d1) / (reps * wl.L)


def step_fraction(wl, ms_step, peaks):
    """The whole step against its roofline: K/V (or I/O) bytes per step for
    the HBM-bound decode steps, FLOPs per step for the tensor-bound ones."""
    if hasattr(wl, "flops"):
        tf = wl.flops() / (ms_step / 1e3) / 1e12
        return {"bound": "tensor", "step_tflops": tf, "step_frac_of_peak": tf / peaks["tensor"][0]}
    gbs = wl.kv_bytes_per_step() / (ms_step / 1e3) / 1e9
    return {"bound": "hbm", "kv_gbs": gbs, "step_frac_of_peak": gbs / peaks["hbm"][0]}


def parity_check(wl, oracle, first_only=False, budget=10.0):
    """Compare the GPU outputs of the timed step with the oracle on a bounded
    sample of whole units (layers, sequences).  Returns (oracle seconds,
    fraction of the step covered, max abs error, units done)."""
    spent, frac, max_err, done = 0.0, 0.0, 0.0, []
    i = 0
    while i < wl.n_samples() and (i == 0 or (not first_only and spent < budget)):
        dt, f, ref, got, what = wl.oracle_sample(i, oracle)
        for k in ref:
            max_err = max(max_err, float(np.abs(got[k] - ref[k]).max()))
        spent += dt
        frac += f
        done.append(what)
        i += 1
    return spent, frac, max_err, done


def measure_config(name, device, steps, warmup, peaks, oracle):
    """One configuration of the headline metric, in this process: step time,
    tokens/s, the step's fraction of its roofline, the dominant kernel's
    fraction, and the oracle's max error on the first unit of the step."""
    import torch
    wl = make_workload(name, device)
    stream = torch.cuda.Stream(device)
    graph = capture_step(wl, stream)
    ms_step = time_graph(graph, stream, steps, warmup) / steps
    launch_ms = time_dominant(wl, stream)
    roof = wl.roofline(launch_ms, peaks)
    _, _, err, done = parity_check(wl, oracle, first_only=True)
    entry = {"ms_per_step": ms_step, "tokens_per_s": wl.tokens_per_step() / (ms_step / 1e3),
             "steps": steps, **step_fraction(wl, ms_step, peaks),
             "dominant_kernel": wl.dominant_kernel, "dominant_launch_us": launch_ms * 1e3,
             "dominant_frac_of_peak": roof["frac"], "dominant_bound": roof["bound"],
             "parity_max_abs_err": err, "parity_checked": f"{done[0]} vs oracle"}
    del graph, wl
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return entry


def config_dict(args, wl, world, kv_bytes):
    return {"workload": args.workload, **{k: v for k, v in wl.cfg.items()},
            "l2": f"inputs larger than L2 ({kv_bytes / 1e9:.2f} GB touched per step "
                  f"vs {L2_BYTES / 1e6:.0f} MB L2)",
            "parallelism": f"replicas x{world} (batch per GPU fixed)",
            "decode_start": ("after the previous launch" if args.no_history_ready else
                             "history ready (asr_set_history_ready: the launches before each "
                             "attention call write none of its lengths or cached rows)")}


def run_ours(args):
    import torch
    import oracle
    from kv_cache_decode_asr_gb300 import build as kbuild
    world, rank, local = dist_setup(args)
    kbuild.build()
    oracle.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    # The decode-attention calls of every workload here are steady decode
    # loops: the launches before each one (another layer's attention or a
    # projection) write none of its lengths, groups or cached rows, so they
    # may read those before the grid dependency wait (asr_set_history_ready).
    from kv_cache_decode_asr_gb300 import ops as kops
    kops.asr_set_history_ready(not args.no_history_ready)
    wl = make_workload(args.workload, device, rank, args.layers)
    if args.separate_append:
        wl.separate_append = True
    if args.separate_reorder:
        wl.separate_reorder = True
    if args.roofline_kernel != "default":
        wl.profile_kernel = args.roofline_kernel
        wl.dominant_kernel = f"roofline of the {args.roofline_kernel} kernel"
    stream = torch.cuda.Stream(device)
    torch.cuda.synchronize()

    # ---- the whole step in one CUDA graph, K replays timed
    graph = capture_step(wl, stream)
    with ClockSampler(local) as clocks:
        ms_total = time_graph(graph, stream, args.steps, args.warmup, world)
    ms_step, value = job_throughput(ms_total, args.steps, wl.tokens_per_step(), world, device)
    tokens = wl.tokens_per_step() * world
    kv_bytes = wl.kv_bytes_per_step()
    kv_gbs = kv_bytes * world / (ms_step / 1e3) / 1e9

    peaks = load_all_peaks()
    launch_ms = time_dominant(wl, stream)
    roof = wl.roofline(launch_ms, peaks)
    roof.update({"traffic": recorded_traffic(wl.kernel_sources, args.workload,
                                             wl.traffic_key()),
                 "kernel": wl.dominant_kernel, "launch_us": launch_ms * 1e3})
    extra = wl.extra_rooflines(stream, peaks) if hasattr(wl, "extra_rooflines") else {}

    cfg_line = config_dict(args, wl, world, kv_bytes)
    gpu_launches = wl.launches() * args.steps

    # ---- end to end through host buffers: per step, H2D of the step's
    # activations from pinned memory, the step, D2H of its outputs
    ins, outs = wl.host_io()
    h_ins = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ins]
    for h, t in zip(h_ins, ins):
        h.copy_(t)
    h_outs = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in ins)
    d2h = sum(t.numel() * t.element_size() for t in outs)
    e2e_steps = max(3, min(args.steps, 50))
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(stream):
        for _ in range(e2e_steps):
            for h, t in zip(h_ins, ins):
                t.copy_(h, non_blocking=True)
            graph.replay()  # the static step graph a caller captures once and replays
            for h, t in zip(h_outs, outs):
                h.copy_(t, non_blocking=True)
    stream.synchronize()
    e2e_s = (time.perf_counter() - t0) / e2e_steps
    e2e_s = max_over_ranks(e2e_s, world, device)
    e2e_value = tokens / e2e_s
    if int(wl.err.item()) != 0:
        raise RuntimeError(f"device error flags {int(wl.err.item()):#x}")

    # ---- CPU oracle on a bounded sample (rank 0, N = 1 only); its outputs
    # double as a parity check of the timed kernels
    cpu = None
    parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        threads = cpu_count()
        oracle.set_threads(threads)
        spent, frac, max_err, done = parity_check(wl, oracle, budget=args.cpu_seconds)
        step_s = spent / frac
        cpu = {"value": wl.tokens_per_step() / step_s, "unit": "tokens/s", "cores": threads,
               "kind": "oracle",
               "sample": f"{len(done)} of {wl.n_samples()} units ({done[0]} .. {done[-1]}), "
                         f"{spent:.1f} s of oracle time, scaled to the whole step"}
        parity = {"max_abs_err": max_err, "checked": f"outputs of {len(done)} units vs oracle",
                  "tolerance": getattr(wl, "parity_tolerance", 2e-3)}
        if hasattr(wl, "parity_note"):
            parity["note"] = wl.parity_note

    # ---- every configuration of the headline metric, same process and box,
    # under one clock record (rank 0 at N = 1, default workload only)
    configs = None
    metric = wl.metric
    if (rank == 0 and world == 1 and not args.no_configs and args.workload == DEFAULT_WORKLOAD
            and not args.layers):
        main_entry = {"ms_per_step": ms_step, "tokens_per_s": value, "steps": args.steps,
                      **step_fraction(wl, ms_step, peaks),
                      "dominant_kernel": wl.dominant_kernel,
                      "dominant_launch_us": launch_ms * 1e3,
                      "dominant_frac_of_peak": roof["frac"], "dominant_bound": roof["bound"],
                      "parity_max_abs_err": parity["max_abs_err"] if parity else None,
                      "parity_checked": parity["checked"] if parity else None,
                      "note": "the main line's own measurement"}
        metric = wl.metric
        del graph, wl
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        oracle.set_threads(cpu_count())
        configs = {}
        with ClockSampler(local) as cclocks:
            for name in CONFIG_WORKLOADS:
                if name == args.workload:
                    configs[name] = main_entry
                else:
                    configs[name] = measure_config(name, device, min(args.steps, 200),
                                                   args.warmup, peaks, oracle)
        configs["clocks"] = cclocks.summary()

    if rank == 0:
        line = {
            "metric": metric,
            "value": value,
            "unit": "tokens/s",
            "n_gpus": world,
            "steps": args.steps,
            "warmup": args.warmup,
            "ms_per_step": ms_step,
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "f16 K/V, fp32 math",
            "data": "synthetic (seeded N(0,1); no weights or audio)",
            "config": cfg_line,
            "kv_gbs": kv_gbs,
            "kv_frac_of_hbm": kv_gbs / world / peaks["hbm"][0],
            "kv_bytes_per_step": kv_bytes,
            "roofline": roof,
            **extra,
            "clocks": clocks.summary(),
            "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                    "step": "the C-ABI calls of one step, captured once as a CUDA graph and "
                            "replayed between the copies"},
            "gpu_launches": gpu_launches,
            "cpu_baseline": cpu,
            "parity": parity,
        }
        if configs is not None:
            line["configs"] = configs
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


# ------------------------------------------------------- reference arm ----

def run_reference(args):
    """The CPU oracle as the reference arm.  Each timed step is one whole
    unit of the workload as the CPU baseline takes it (one layer of every
    sequence; one sequence of a prefill), so `steps` x `ms_per_step` is the
    oracle time actually spent; `value` scales a unit to the whole step."""
    world, rank, local = dist_setup(args)
    if rank != 0:
        return
    import torch
    import oracle
    oracle.build()
    threads = cpu_count()
    oracle.set_threads(threads)
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    wl = make_workload(args.workload, device, 0, args.layers) if device.type == "cuda" else None
    if wl is None:
        print(json.dumps({"impl": "reference", "unavailable": "needs the device-drawn inputs"}))
        return
    n = wl.n_samples()
    for i in range(args.warmup):
        wl.oracle_sample(i % n, oracle)
    times, fracs = [], []
    for i in range(args.steps):
        dt, f, _, _, _ = wl.oracle_sample((args.warmup + i) % n, oracle)
        times.append(dt)
        fracs.append(f)
    unit_s = sum(times) / len(times)
    step_s = sum(times) / sum(fracs)
    value = wl.tokens_per_step() / step_s
    kv_bytes = wl.kv_bytes_per_step()
    line = {
        "impl": "reference",
        "metric": wl.metric,
        "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": unit_s * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded N(0,1); no weights or audio)",
        "config": config_dict(args, wl, world, kv_bytes),
        "units_per_workload_step": round(1.0 / (sum(fracs) / len(fracs)), 3),
        "workload_step_ms": step_s * 1e3,
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle",
                         "sample": f"each timed step is one whole unit of the workload "
                                   f"({n} units make one workload step; "
                                   f"ms_per_step is the oracle time of one unit)"},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(syn.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-configuration measurements of the default line")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-history-ready", action="store_true",
                    help="decode-attention calls wait for the previous launch before reading "
                         "their lengths and history (the library's default order)")
    ap.add_argument("--separate-reorder", action="store_true",
                    help="beam workload: one asr_kv_rearrange launch before the layers instead "
                         "of the reorder fused into each layer's append + self launch")
    ap.add_argument("--separate-append", action="store_true",
                    help="Whisper: launch the K/V append and the self-attention separately")
    ap.add_argument("--roofline-kernel", default="default", choices=["default", "cross", "self"],
                    help="Whisper: which kernel the roofline object times (default: cross)")
    ap.add_argument("--layers", type=int, default=0,
                    help="run fewer layers than the model has (small cases for profiling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()

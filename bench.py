#!/usr/bin/env python
"""Throughput of speculative-decoding verification on GB300.

One step = one call of the verification path over one batch of synthetic
logits already resident in HBM (the workload's whole hot path: for the EAGLE
tree workloads that is the tree mask plus tree verification, for eagle2 also
expand + rerank).  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                  [--impl ours|reference]

Multi-GPU (torchrun, one rank per GPU): every rank verifies its own batch
(sequences are independent, no collective on the data path); the time is the
max over ranks and the value counts the rows of all ranks (weak scaling).

--impl reference times the float64 CPU oracle (tests' ground truth) on a
bounded sample of the same workload on the host cores.
"""

from __future__ import annotations

import os

# the CPU legs time the oracle on one thread (numpy's BLAS included)
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse
import json
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "verified draft rows/s at V=128256"
UNIT = "rows/s"
DEFAULT_WORKLOAD = "tree_static"


def _args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD,
                   choices=["tree_static", "greedy", "eagle2", "chain_topk",
                            "chain_sample", "lmhead_tree", "kv_commit",
                            "accept_stats", "tree_attention"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--cpu-seconds", type=float, default=12.0)
    p.add_argument("--B", type=int, default=None,
                   help="override the workload's batch (small profiling "
                        "cases); the default is the workload's own batch")
    p.add_argument("--no-extend", action="store_true",
                   help="do not keep the load running for the clock sampler "
                        "after a short timed region (profiler runs)")
    p.add_argument("--no-configs", action="store_true",
                   help="time the chosen workload only (by default the "
                        "tree_static line also times the other "
                        "verification workloads under its `configs` key)")
    return p.parse_args()


# Verification workloads timed beside the headline one (each is one of the
# pages' configurations; see synth.workload).
OTHER_CONFIGS = ("greedy", "eagle2", "chain_topk", "chain_sample",
                 "lmhead_tree")
L2_BYTES = 129 * 2**20  # GB300 L2 (about 129 MB)


def metric_of(w):
    return f"verified draft rows/s at V={w.V}"


# DRAM traffic per launch of the profiled kernel, from one ncu capture
# (dram__bytes_read.sum + dram__bytes_write.sum of a smaller batch, scaled
# to the rows the kernel processes), keyed by workload, with a hash of the
# sources the kernel is built from at capture time (and of the header
# definitions they use).  Reported as null once they changed.
_STREAM_SRC = ("sample_stream.cuh", "sample_stream_bf16.cu",
               "sample_stream_f32.cu", "common.cuh", "kernels.h")
TRAFFIC = {
    # unit_stream, tree_static at B=16 (clusters of 2): 761.82 MB read +
    # 3.03 MB written, 976 rows
    "tree_static": {"bytes_per_unit": 764.85e6 / 976, "src": _STREAM_SRC,
                    "hash": "e18c07afe65b4561"},
    # unit_stream, eagle2 at B=32 (one CTA per row): 402.91 MB read + 3.17 MB
    # written, 782 rows with a draft row
    "eagle2": {"bytes_per_unit": 406.08e6 / 782, "src": _STREAM_SRC,
               "hash": "e18c07afe65b4561"},
    # accept_stats_warp at B=65536 rounds: 47.46 MB read + 6.9 KB written
    "accept_stats": {"bytes_per_unit": 47.47e6 / 65536,
                     "src": ("accept_stats.cu", "common.cuh", "kernels.h"),
                     "hash": "fcd87afa19a48919"},
}


def _src_hash(files):
    """Hash of a kernel's sources and of the parts of the public header they
    use (the #define constants and typedef structs they name), so that
    declarations and comments added for other entry points do not count as
    a change of this kernel."""
    import hashlib
    import re
    d = os.path.join(ROOT, "speculative_decoding_verification_tree_gb300",
                     "csrc")
    h = hashlib.sha256()
    texts = []
    for f in files:
        try:
            with open(os.path.join(d, f), "rb") as fh:
                data = fh.read()
            h.update(f.encode() + b"\0" + data)
            texts.append(data.decode("utf-8", "replace"))
        except OSError:
            h.update(f.encode() + b"\0missing")
    with open(os.path.join(ROOT, "include", "specverify.h"),
              encoding="utf-8") as fh:
        hdr = re.sub(r"/\*.*?\*/", "", fh.read(), flags=re.S)
    used = set(re.findall(r"\b(?:SPEC_[A-Z0-9_]+|spec_\w+_t)\b",
                          "".join(texts)))
    for m in re.finditer(r"#define\s+(\w+)[^\n]*", hdr):
        if m.group(1) in used:
            h.update(m.group(0).encode())
    # typedef struct {...} name; and typedef struct tag {...} name;
    for m in re.finditer(r"typedef\s+struct\s*(\w+)?\s*\{.*?\}\s*(\w+)\s*;",
                         hdr, flags=re.S):
        if m.group(2) in used or (m.group(1) and m.group(1) in used):
            h.update(m.group(0).encode())
    return h.hexdigest()[:16]


def _traffic(name, units):
    t = TRAFFIC.get(name)
    if not t or t["hash"] != _src_hash(t["src"]):
        return None
    return int(t["bytes_per_unit"] * units)


def _tensor_peak():
    """Dense bf16 tensor peak (TFLOP/s) for a kernel timed inside a long
    step: the measured sustained figure, else the fallback."""
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops_sustained"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1700.0, "fallback"


def roofline_of(work, kern_ms, peak, peak_kind, rc, name):
    """Roofline object of the step's dominant kernel."""
    if work.bound == "tensor":
        tpk, tkind = _tensor_peak()
        tf = work.kernel_flops / (kern_ms / 1e3) / 1e12
        return {"bound": "tensor", "achieved": round(tf, 1), "peak": tpk,
                "unit": "TFLOP/s", "frac": round(tf / tpk, 4),
                "traffic": _traffic(name, work.kernel_units),
                "kernel": work.kernel_name,
                "flops_per_launch": work.kernel_flops,
                "bytes_per_launch": work.kernel_bytes,
                "avg_launch_ms": round(kern_ms, 5),
                "peak_source": f"{tkind} (bf16_tflops_sustained)",
                "profile_rc": rc}
    achieved = work.kernel_bytes / (kern_ms / 1e3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
            "unit": "GB/s", "frac": round(achieved / peak, 4),
            "traffic": _traffic(name, work.kernel_units),
            "kernel": work.kernel_name,
            "bytes_per_launch": work.kernel_bytes,
            "avg_launch_ms": round(kern_ms, 5), "peak_source": peak_kind,
            "profile_rc": rc}


def verify_kernel(h, lib, work, peak):
    """The verification kernel's share beside an LM-head GEMM."""
    vms, nv, _ = kernel_time(h, lib.SPEC_PROF_VERIFY)
    if not nv:
        return {}
    gbs = work.verify_bytes / (vms / 1e3) / 1e9
    return {"unit_stream": {"avg_launch_ms": round(vms, 5),
                            "bytes_per_launch": work.verify_bytes,
                            "achieved_gbs": round(gbs, 1),
                            "frac": round(gbs / peak, 4)}}


def _peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def _chain_single_launch(B, K, V, tsz, dsz, device):
    """Whether the library verifies this sampled chain (no truncation) in
    its single-launch form: 1 <= K <= 16, V a multiple of 8, one 8-CTA
    cluster per sequence within one wave of the GPU's SMs, and each CTA's
    eighth of the K + 1 target and K draft rows within 200 KB of shared
    memory."""
    import torch
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    if not (1 <= K <= 16) or V % 8 or B * 8 > sms:
        return False
    sl = ((V + 7) // 8 + 7) // 8 * 8
    return (K + 1) * sl * tsz + K * sl * dsz <= 200 * 1024


# ------------------------------------------------------------- workloads
class Work:
    """Device inputs, outputs and one step of a workload (GPU arm)."""

    def __init__(self, name, device, B=None):
        import torch

        import synth
        from speculative_decoding_verification_tree_gb300 import _lib, api
        self.torch, self.api, self.lib = torch, api, _lib
        self.name = name
        self.w = w = (synth.workload(name) if B is None else
                      synth.workload(name, B=B))
        self.device = device
        if name in ("greedy", "chain_topk", "chain_sample"):
            self.kind = "chain"
            self.target, self.draft, self.toks = synth.chain_inputs(w, device)
            B, K, V = w.B, w.K, w.V
            self.rows = B * K
            self.kernel_units = self.rows
            self.ws = api.workspace(_lib.SPEC_OP_CHAIN, B, K, V, device)
            self.out = (torch.empty(B, dtype=torch.int32, device=device),
                        torch.empty(B, K + 1, dtype=torch.int32, device=device),
                        torch.empty(B, K, dtype=torch.float32, device=device))
            self.inputs = [self.target, self.draft, self.toks]
            self.prof_kind = (_lib.SPEC_PROF_ARGMAX if w.temperature == 0
                              else _lib.SPEC_PROF_VERIFY)
            # the profiled launch: the argmax pass (greedy), the candidate
            # top-k pass (top-k / top-p sampling) or the full-row pipeline
            self.kernel_name = ("argmax_partial" if w.temperature == 0 else
                                "topk_rows" if (w.top_k > 0 or w.top_p < 1)
                                else "unit_stream")
            tb = self.target.element_size()
            self.kernel_bytes = B * (K + 1) * V * tb
            if w.temperature > 0:
                self.kernel_bytes += B * K * V * self.draft.element_size()
            # argmax + finalize; top-k rows (with the row records) and the
            # candidate-list verification (with the walk); or records,
            # streaming verification, walk
            self.launches_per_step = (2 if w.temperature == 0 else
                                      2 if (w.top_k > 0 or w.top_p < 1)
                                      else 3)
            if w.temperature > 0 and w.top_k == 0 and w.top_p >= 1 and \
                    _chain_single_launch(B, K, V, tb,
                                         self.draft.element_size(), device):
                # one cluster of 8 CTAs per sequence, every row resident in
                # shared memory: a single launch
                self.kernel_name = "chain_small"
                self.launches_per_step = 1
        elif name == "tree_static":
            self.kind = "tree"
            (self.target, self.draft, self.q_row, self.toks,
             self.parent) = synth.tree_inputs(w, device)
            B, N, V = w.B, self.toks.shape[1], w.V
            self.N = N
            self.rows = B * (N + 1)
            self.kernel_units = self.rows
            self.ws = api.workspace(_lib.SPEC_OP_TREE, B, N, V, device)
            self.out = (torch.empty(B, dtype=torch.int32, device=device),
                        torch.empty(B, N, dtype=torch.int32, device=device),
                        torch.empty(B, N + 1, dtype=torch.int32, device=device),
                        torch.empty(B, N + 1, dtype=torch.float32,
                                    device=device))
            self.mask = torch.empty(B, N, N, dtype=torch.uint8, device=device)
            self.inputs = [self.target, self.draft, self.q_row, self.toks,
                           self.parent]
            self.prof_kind = _lib.SPEC_PROF_VERIFY
            self.kernel_name = ("topk_rows" if (w.top_k > 0 or w.top_p < 1)
                                else "unit_stream")
            self.kernel_bytes = B * (N + 1) * V * (
                self.target.element_size() + self.draft.element_size())
            # mask, row records, row verification, walk (top-k / top-p:
            # mask, top-k rows with the records, candidate-list verification
            # with the walk)
            self.launches_per_step = (3 if (w.top_k > 0 or w.top_p < 1)
                                      else 4)
        elif name == "eagle2":
            self.kind = "eagle2"
            self.draft = synth.eagle2_draft(w, device)
            B, V, M = w.B, w.V, w.total
            self.N = M
            self.R = self.draft.shape[1]
            self.ews = api.workspace(_lib.SPEC_OP_EAGLE2, B, self.R, V, device)
            # each draft row's log2 normaliser: written by the expand, read
            # by the verification (which then skips summing the draft rows)
            self.lse = torch.empty(B, self.R, dtype=torch.float32,
                                   device=device)
            self.tree = (torch.empty(B, M, dtype=torch.int32, device=device),
                         torch.empty(B, M, dtype=torch.int32, device=device),
                         torch.empty(B, M + 1, dtype=torch.int32,
                                     device=device),
                         torch.empty(B, M, dtype=torch.float32, device=device),
                         torch.empty(B, M, M, dtype=torch.uint8,
                                     device=device))
            self._expand(self.draft)
            torch.cuda.synchronize()
            # target rows for the reranked tree (synthetic target forward)
            self.target = synth.eagle2_target(w, self.draft, self.tree[2],
                                              device)
            self.rows = B * (M + 1)
            self.ws = api.workspace(_lib.SPEC_OP_TREE, B, M, V, device)
            self.out = (torch.empty(B, dtype=torch.int32, device=device),
                        torch.empty(B, M, dtype=torch.int32, device=device),
                        torch.empty(B, M + 1, dtype=torch.int32, device=device),
                        torch.empty(B, M + 1, dtype=torch.float32,
                                    device=device))
            self.inputs = [self.draft, self.target]
            self.prof_kind = _lib.SPEC_PROF_VERIFY
            self.kernel_name = "unit_stream"
            # unit_stream reads the target and draft row of every node that
            # has a draft row; a target row without one is read by the walk,
            # and only when the accepted path ends there
            qrows = int((self.tree[2] >= 0).sum().item())
            self.kernel_units = qrows
            self.kernel_bytes = qrows * V * (2 + 2)
            self.expand_bytes = B * self.R * V * 2
            # expand rows, select, mask, row records, verification, walk
            self.launches_per_step = 6
        elif name == "lmhead_tree":
            # the static tree with the target logits from the LM head
            self.kind = "lmhead"
            (self.hidden, self.wv, self.draft, self.q_row, self.toks,
             self.parent) = synth.lmhead_tree_inputs(w, device)
            B, N, V, H = w.B, self.toks.shape[1], w.V, w.H
            self.N = N
            self.rows = B * (N + 1)
            self.kernel_units = self.rows
            self.ws = api.workspace(_lib.SPEC_OP_TREE_LMHEAD, B, N, V, device)
            self.out = (torch.empty(B, dtype=torch.int32, device=device),
                        torch.empty(B, N, dtype=torch.int32, device=device),
                        torch.empty(B, N + 1, dtype=torch.int32, device=device),
                        torch.empty(B, N + 1, dtype=torch.float32,
                                    device=device))
            self.mask = torch.empty(B, N, N, dtype=torch.uint8, device=device)
            self.inputs = [self.hidden, self.wv, self.draft, self.q_row,
                           self.toks, self.parent]
            self.resident = {1}  # the LM head's weights stay in HBM
            self.prof_kind = _lib.SPEC_PROF_LMHEAD
            self.kernel_name = "lmhead_gemm"
            self.bound = "tensor"
            self.kernel_flops = 2 * self.rows * H * V
            # reads hidden and W, writes the bf16 logits
            self.kernel_bytes = (self.rows * H + V * H + self.rows * V) * 2
            # the verifier then reads the logits and draft rows once each
            self.verify_bytes = self.rows * V * (2 + self.draft.element_size())
            # mask, GEMM, normaliser merge, row records, verification, walk
            self.launches_per_step = 6
        else:
            raise SystemExit(f"workload {name} is not wired into the bench")

    def input_bytes(self):
        """Bytes of the step's device inputs (decides the L2 flush)."""
        return sum(x.numel() * x.element_size() for x in self.inputs
                   if x is not None)

    def _expand(self, draft):
        w = self.w
        self.api.spec_eagle2_expand_rerank(
            draft, temperature=w.temperature, depth=w.depth, topk=w.topk,
            width=w.width, total=w.total, out=self.tree, ws=self.ews,
            draft_lse=self.lse)

    def step(self, inputs=None):
        """Enqueue one step on the current stream."""
        api, w = self.api, self.w
        x = self.inputs if inputs is None else inputs
        if self.kind == "chain":
            api.spec_verify_chain(x[0], x[1], x[2], temperature=w.temperature,
                                  top_k=w.top_k, top_p=w.top_p,
                                  draft_kind=w.draft_kind,
                                  seed=w.decision_seed, out=self.out,
                                  ws=self.ws)
        elif self.kind == "eagle2":
            self._expand(x[0])
            tok, par, qrow = self.tree[0], self.tree[1], self.tree[2]
            api.spec_verify_tree(x[1], x[0], qrow, tok, par,
                                 temperature=w.temperature,
                                 seed=w.decision_seed, out=self.out,
                                 ws=self.ws, draft_lse=self.lse)
        elif self.kind == "lmhead":
            from speculative_decoding_verification_tree_gb300.api import (
                _ptr, _stream)
            B, N = self.w.B, self.N
            self.lib.call("spec_tree_mask", _ptr(x[5]), B, N, _ptr(self.mask),
                          None, _stream(None))
            api.spec_verify_tree_lmhead(x[0], x[1], x[2], x[3], x[4], x[5],
                                        temperature=w.temperature,
                                        draft_kind=w.draft_kind,
                                        seed=w.decision_seed, out=self.out,
                                        ws=self.ws)
        else:
            from speculative_decoding_verification_tree_gb300.api import (
                _ptr, _stream)
            B, N = self.w.B, self.N
            self.lib.call("spec_tree_mask", _ptr(x[4]), B, N, _ptr(self.mask),
                          None, _stream(None))
            api.spec_verify_tree(x[0], x[1], x[2], x[3], x[4],
                                 temperature=w.temperature, top_k=w.top_k,
                                 top_p=w.top_p, draft_kind=w.draft_kind,
                                 seed=w.decision_seed, out=self.out,
                                 ws=self.ws)

    bound = "hbm"
    resident = frozenset()

    def host_copy(self):
        """The step's inputs on the host, for the CPU oracle."""
        if self.kind == "lmhead":
            keys = ["hidden", "w", "draft", "q_row", "toks", "parent"]
            return self.w, {k: x.cpu() for k, x in zip(keys, self.inputs)}
        if self.kind == "eagle2":
            return self.w, {"draft": self.draft.cpu(),
                            "target": self.target.cpu()}
        keys = (["target", "draft", "toks"] if self.kind == "chain" else
                ["target", "draft", "q_row", "toks", "parent"])
        return self.w, {k: (None if x is None else x.cpu())
                        for k, x in zip(keys, self.inputs)}

    def outputs(self):
        if self.kind == "eagle2":
            return list(self.out) + list(self.tree)
        return [o for o in self.out if o is not None]

    def emitted_tokens(self):
        return int(self.out[0].sum().item()) + self.w.B


# ------------------------------------------------------------------ clocks
class Clocks:
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100", "-i",
                 str(self.index)], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
            self.t0 = time.time()
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        # under load: drop idle samples at the edges of the window
        top = max(sm)
        load = [x for x in sm if x >= 0.5 * top] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# -------------------------------------------------------------- CPU oracle
def oracle_step(w, host, seqs):
    """Run the oracle on sequences `seqs` of the host copy of the inputs."""
    import numpy as np
    from oracle.chain import verify_chain
    from oracle.eagle2 import expand_rerank
    from oracle.tree import tree_mask, verify_tree
    if w.name == "lmhead_tree":
        from oracle.lmhead import verify_tree_lmhead
        if "w64" not in host:  # the LM head in float64, converted once
            host["w64"] = host["w"].float().numpy().astype(np.float64)
        par = host["parent"][seqs].numpy()
        res = verify_tree_lmhead(
            host["hidden"][seqs].float().numpy().astype(np.float64),
            host["w64"], host["draft"][seqs].float().numpy().astype(
                np.float64), host["q_row"][seqs].numpy(),
            host["toks"][seqs].numpy(), par, temperature=w.temperature,
            draft_kind=w.draft_kind, seed=w.decision_seed, batch_ids=seqs)
        return len(seqs) * (par.shape[1] + 1), res.ref
    t = host["target"][seqs].float().numpy().astype(np.float64)
    if w.name == "eagle2":
        d = host["draft"][seqs].float().numpy().astype(np.float64)
        tr = expand_rerank(d, temperature=w.temperature, depth=w.depth,
                           topk=w.topk, width=w.width, total=w.total)
        ref = verify_tree(t, d, tr.q_row, tr.node_tokens, tr.parent,
                          temperature=w.temperature, seed=w.decision_seed,
                          batch_ids=seqs)
        return len(seqs) * (w.total + 1), (tr, ref)
    if w.name in ("greedy", "chain_topk", "chain_sample"):
        d = None if host["draft"] is None else \
            host["draft"][seqs].float().numpy().astype(np.float64)
        ref = verify_chain(t, d, host["toks"][seqs].numpy(),
                           temperature=w.temperature, top_k=w.top_k,
                           top_p=w.top_p, draft_kind=w.draft_kind,
                           seed=w.decision_seed, batch_ids=seqs)
        return len(seqs) * w.K, ref
    d = host["draft"][seqs].float().numpy().astype(np.float64)
    par = host["parent"][seqs].numpy()
    tree_mask(par)
    ref = verify_tree(t, d, host["q_row"][seqs].numpy(),
                      host["toks"][seqs].numpy(), par,
                      temperature=w.temperature, top_k=w.top_k,
                      top_p=w.top_p, draft_kind=w.draft_kind,
                      seed=w.decision_seed, batch_ids=seqs)
    return len(seqs) * (par.shape[1] + 1), ref


def host_inputs(name, nseq=8):
    """The first `nseq` sequences of the workload's shape, generated on the
    host (CPU generator); the oracle is timed per sequence."""
    import synth
    w = synth.workload(name)
    w = synth.workload(name, B=min(w.B, nseq))
    if name in ("greedy", "chain_topk", "chain_sample"):
        t, d, k = synth.chain_inputs(w, "cpu")
        return w, {"target": t, "draft": d, "toks": k}
    if name == "lmhead_tree":
        hd, wv, d, q, k, p = synth.lmhead_tree_inputs(w, "cpu")
        return w, {"hidden": hd, "w": wv, "draft": d, "q_row": q, "toks": k,
                   "parent": p}
    if name == "eagle2":
        import torch
        d = synth.eagle2_draft(w, "cpu")
        # host-side stand-in for the target forward of the reranked tree:
        # tree row r reuses draft row r where it exists (the oracle's cost
        # does not depend on which rows these are)
        R = d.shape[1]
        r = torch.arange(w.total + 1, dtype=torch.int32)
        q_row = torch.where(r < R, r, torch.full_like(r, -1))
        q_row = q_row.unsqueeze(0).expand(w.B, -1).contiguous()
        return w, {"draft": d, "target": synth.eagle2_target(w, d, q_row,
                                                              "cpu")}
    t, d, q, k, p = synth.tree_inputs(w, "cpu")
    return w, {"target": t, "draft": d, "q_row": q, "toks": k, "parent": p}


def time_oracle(name, seconds, host=None, results=None):
    """Oracle rows/s on a bounded sample: sequences one by one until
    `seconds` of CPU work.  `results` (a list) receives (b, oracle result)
    per sequence."""
    w, host = host_inputs(name) if host is None else host
    rows, t0, b = 0, time.perf_counter(), 0
    while True:
        r, ref = oracle_step(w, host, [b % w.B])
        rows += r
        if results is not None:
            results.append((b % w.B, ref))
        b += 1
        el = time.perf_counter() - t0
        if el >= seconds or b >= w.B:
            break
    return rows / el, b, el


def parity_counts(work, results):
    """Compare the GPU outputs of the timed step with the oracle results of
    the sampled sequences: compared element by element (exact, or a final
    draw inside the 1e-5 CDF band), excluded as near ties (an accept test
    within 1e-5 of its threshold), and mismatches (must be 0)."""
    import numpy as np
    out = [o.cpu().numpy() for o in work.out]
    c = {"sequences": 0, "compared": 0, "exact": 0, "near_tie_excluded": 0,
         "cdf_band": 0, "mismatch": 0}
    for b, ref in results:
        c["sequences"] += 1
        if work.kind == "eagle2":
            tr, ref = ref
            tree = [t.cpu().numpy() for t in work.tree]
            if not (np.array_equal(tree[0][b], tr.node_tokens[0]) and
                    np.array_equal(tree[1][b], tr.parent[0])):
                c["mismatch"] += 1  # reranked tree differs
                continue
        if ref.near_tie[0]:
            c["near_tie_excluded"] += 1
            continue
        c["compared"] += 1
        if work.kind == "chain":
            n = int(ref.accepted[0])
            same = int(out[0][b]) == n
            tok = out[1][b]
        else:
            n = int(ref.path_len[0])
            same = (int(out[0][b]) == n and
                    np.array_equal(out[1][b], ref.path_nodes[0]))
            tok = out[2][b]
        same = (same and np.array_equal(tok[:n], ref.tokens[0][:n]) and
                np.array_equal(tok[n + 1:], ref.tokens[0][n + 1:]))
        if not same:
            c["mismatch"] += 1
        elif tok[n] == ref.tokens[0][n]:
            c["exact"] += 1
        elif ref.sample_near is not None and ref.sample_near[0]:
            c["cdf_band"] += 1
        else:
            c["mismatch"] += 1
    return c


def cpu_sample_text(name, nseq, el):
    return (f"{nseq} of the workload's sequences, one by one, "
            f"{el:.1f} s of single-thread numpy float64")


# ------------------------------------------------------------------- main
def max_over_ranks(dist, ms, dev):
    """The slowest rank's time (every rank gets it); `dist` None = 1 rank."""
    if not dist:
        return ms
    import torch
    t = torch.tensor([float(ms)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, steps, world, ms):
    """Whole-job throughput: the units all ranks processed / the time."""
    return units_per_rank * steps * world / (ms / 1e3)


def spawn_ranks(args):
    """`--gpus N` outside torchrun: launch N local ranks (one per GPU)
    through torch.distributed.run on 127.0.0.1 and return their exit code;
    rank 0 prints the line."""
    import socket
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
           f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
           "--master-port", str(port), os.path.abspath(__file__),
           *sys.argv[1:]]
    return subprocess.call(cmd)


def time_steps(torch, work, steps, flush=None):
    """Enqueue `steps` steps and return the summed device time (ms) of the
    steps alone.  With `flush` (a buffer larger than L2) every step is
    preceded by a write of the whole buffer, outside the timed events, so
    each step starts with the inputs out of L2, and by a device-side spin
    that keeps the GPU's queue ahead of the host."""
    if flush is None:
        ev0 = torch.cuda.Event(enable_timing=True)
        ev1 = torch.cuda.Event(enable_timing=True)
        ev0.record()
        for _ in range(steps):
            work.step()
        ev1.record()
        torch.cuda.synchronize()
        return ev0.elapsed_time(ev1)
    evs = []
    for _ in range(steps):
        flush.zero_()
        # a short spin on the device (outside the events) keeps the GPU's
        # queue ahead of the host, so that the events time the step on the
        # device rather than the host enqueueing it (the host's part of a
        # call is in the e2e figure)
        torch.cuda._sleep(100000)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record()
        work.step()
        e1.record()
        evs.append((e0, e1))
    torch.cuda.synchronize()
    return sum(e0.elapsed_time(e1) for e0, e1 in evs)


# The dominant kernel is timed on every PROFILE_EVERY-th launch in the timed
# region (its event pair costs about 4 us of device time on the step it
# brackets, which would inflate short steps if taken every time).
PROFILE_EVERY = 4


def kernel_time(h, kind):
    """(average launch ms, launches, rc) of one profiled kernel kind."""
    import ctypes
    tot, nl = ctypes.c_double(0), ctypes.c_int(0)
    rc = h.spec_profile_read(kind, ctypes.byref(tot), ctypes.byref(nl))
    return (tot.value / nl.value if nl.value else None), nl.value, rc


def l2_note(work):
    return ("inputs exceed L2 (no flush)" if work.input_bytes() > L2_BYTES
            else "L2 flushed before every timed step (2 x L2 written "
                 "outside the timed events)")


def run_config(torch, h, lib, name, dev, steps, peak, peak_kind):
    """Time one more verification workload; returns its summary (step time,
    dominant kernel and its fraction of the HBM roofline)."""
    work = Work(name, dev)
    flush = None
    if work.input_bytes() <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(5):
        work.step()
    torch.cuda.synchronize()
    h.spec_profile_enable(PROFILE_EVERY)
    ms = time_steps(torch, work, steps, flush)
    kern_ms, nl, rc = kernel_time(h, work.prof_kind)
    other = {}
    if work.kind == "lmhead":
        other["unit_stream"] = verify_kernel(h, lib, work, peak).get(
            "unit_stream")
    if work.kind == "eagle2":
        ems, n2, _ = kernel_time(h, lib.SPEC_PROF_EXPAND)
        if n2:
            other["eagle2_rows"] = {
                "avg_launch_ms": round(ems, 5),
                "bytes_per_launch": work.expand_bytes,
                "frac": round(work.expand_bytes / (ems / 1e3) / 1e9 / peak,
                              4)}
    h.spec_profile_enable(0)
    w = work.w
    d = {"metric": metric_of(w), "unit": UNIT,
         "value": round(work.rows * steps / (ms / 1e3), 1),
         "ms_per_step": round(ms / steps, 5), "steps": steps,
         "B": w.B, "drafts_per_seq": w.K, "V": w.V,
         "temperature": w.temperature, "dtype": dtype_name(w),
         "l2": l2_note(work), "kernel": work.kernel_name,
         "avg_launch_ms": None if kern_ms is None else round(kern_ms, 5),
         "bytes_per_launch": work.kernel_bytes, "profile_rc": rc,
         "gpu_launches": work.launches_per_step * steps}
    if kern_ms and work.bound == "tensor":
        r = roofline_of(work, kern_ms, peak, peak_kind, rc, name)
        d.update({"bound": "tensor", "achieved_tflops": r["achieved"],
                  "peak_tflops": r["peak"], "peak_source": r["peak_source"],
                  "frac": r["frac"], "flops_per_launch": work.kernel_flops})
        d["other_kernels"] = verify_kernel(h, lib, work, peak)
    elif kern_ms:
        gbs = work.kernel_bytes / (kern_ms / 1e3) / 1e9
        d.update({"achieved_gbs": round(gbs, 1), "peak_gbs": peak,
                  "peak_source": peak_kind, "frac": round(gbs / peak, 4)})
    if work.kind == "eagle2":
        step_bytes = work.kernel_bytes + work.expand_bytes
        d["step_frac"] = round(step_bytes / (ms / steps / 1e3) / 1e9 / peak,
                               4)
        d["other_kernels"] = other
    d["tokens_per_s"] = round(work.emitted_tokens() * steps / (ms / 1e3), 1)
    del work, flush
    torch.cuda.empty_cache()
    return d


def workload_config(name, w, world):
    return {"workload": name, "B": w.B, "drafts_per_seq": w.K, "V": w.V,
            "temperature": w.temperature, "top_k": w.top_k,
            "top_p": w.top_p,
            "parallelism": f"replicas x{world} (sequences split)"}


def main():
    args = _args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        return spawn_ranks(args)
    if args.gpus != world:
        raise SystemExit(f"--gpus {args.gpus} but WORLD_SIZE={world}: launch "
                         "one rank per GPU (or leave WORLD_SIZE unset)")

    if args.workload == "kv_commit":
        return kv_main(args, world, rank, local)
    if args.workload == "accept_stats":
        return stats_main(args, world, rank, local)
    if args.workload == "tree_attention":
        return attn_main(args, world, rank, local)
    if args.impl == "reference":
        return reference_arm(args, world, rank)

    import torch
    import __graft_entry__ as g
    g.build()
    from speculative_decoding_verification_tree_gb300 import _lib
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    work = Work(args.workload, dev, args.B)
    steps = args.steps or (3000 if args.workload != "eagle2" else 800)
    warm = max(3, args.warmup)
    flush = None
    if work.input_bytes() <= L2_BYTES:
        flush = torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(warm):
        work.step()
    torch.cuda.synchronize()

    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    h = _lib.load()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    h.spec_profile_enable(PROFILE_EVERY)
    ms = time_steps(torch, work, steps, flush)
    if dist:
        dist.barrier()
    kern_ms, nl, rc = kernel_time(h, work.prof_kind)
    peak, peak_kind = _peaks()
    other = {}
    if work.kind == "lmhead":
        other = verify_kernel(h, _lib, work, peak)
    if work.kind == "eagle2":
        ems_k, n2, _ = kernel_time(h, _lib.SPEC_PROF_EXPAND)
        if n2:
            other["eagle2_rows"] = {
                "avg_launch_ms": round(ems_k, 5),
                "bytes_per_launch": work.expand_bytes,
                "achieved_gbs": round(work.expand_bytes / (ems_k / 1e3) / 1e9,
                                      1)}
    h.spec_profile_enable(0)
    t_region = ms / 1e3
    if t_region < 1.0 and not args.no_extend:
        # keep the clock sampler running on the same load
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for _ in range(50):
                work.step()
            torch.cuda.synchronize()
    clocks.stop()
    ms = max_over_ranks(dist, ms, dev)
    ms_step = ms / steps
    value = job_rate(work.rows, steps, world, ms)
    tokens_per_step = work.emitted_tokens()

    roof = None
    if kern_ms:
        roof = roofline_of(work, kern_ms, peak, peak_kind, rc, args.workload)
        roof["other_kernels"] = other

    # end to end through the public API from pinned host buffers
    e2e = None
    if not args.no_e2e:
        # inputs resident in HBM across steps (model weights) are not copied
        host_in = [None if (x is None or i in work.resident) else
                   x.cpu().pin_memory() for i, x in enumerate(work.inputs)]
        dev_in = [x if i in work.resident else
                  (None if x is None else torch.empty_like(x))
                  for i, x in enumerate(work.inputs)]
        host_out = [o.cpu().pin_memory() for o in work.outputs()]
        h2d = sum(x.numel() * x.element_size() for x in host_in
                  if x is not None)
        d2h = sum(x.numel() * x.element_size() for x in host_out)
        n_e2e = max(3, min(steps, 20))

        def e2e_step():
            for d, s in zip(dev_in, host_in):
                if d is not None and s is not None:
                    d.copy_(s, non_blocking=True)
            work.step(dev_in)
            for d, s in zip(host_out, work.outputs()):
                d.copy_(s, non_blocking=True)
        e2e_step()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(n_e2e):
            e2e_step()
        a1.record()
        torch.cuda.synchronize()
        ems = a0.elapsed_time(a1)
        ems = max_over_ranks(dist, ems, dev)
        e2e = {"value": round(job_rate(work.rows, n_e2e, world, ems), 1),
               "unit": UNIT, "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "steps": n_e2e,
               "ms_per_step": round(ems / n_e2e, 4)}

    cpu = parity = None
    if rank == 0 and world == 1 and not args.no_cpu:
        results = []
        rps, nseq, el = time_oracle(args.workload, args.cpu_seconds,
                                    work.host_copy(), results)
        cpu = {"value": round(rps, 2), "unit": UNIT, "cores": 1,
               "kind": "oracle",
               "sample": cpu_sample_text(args.workload, nseq, el)}
        # the same sequences' GPU outputs against the oracle's
        parity = parity_counts(work, results)
        parity["rule"] = ("decisions exact except an accept test within "
                          "1e-5 of its threshold (excluded, counted); a "
                          "final draw may differ only inside the 1e-5 CDF "
                          "band (counted)")

    rows_per_step, launches, l2 = work.rows, work.launches_per_step, \
        l2_note(work)
    configs = None
    if (args.workload == DEFAULT_WORKLOAD and args.B is None and
            not args.no_configs):
        w0 = work.w
        del work, flush
        torch.cuda.empty_cache()
        configs = {}
        cclk = Clocks(local)
        cclk.start()
        for name in OTHER_CONFIGS:
            n = {"greedy": 1000, "eagle2": 300, "chain_topk": 500,
                 "chain_sample": 500, "lmhead_tree": 100}[name]
            if args.steps is not None:  # short runs (profiler captures)
                n = max(10, min(n, args.steps))
            configs[name] = run_config(torch, h, _lib, name, dev, n, peak,
                                       peak_kind)
        n = 300 if args.steps is None else max(10, min(300, args.steps))
        configs["tree_attention"] = attn_config(torch, h, _lib, dev, n, peak,
                                                peak_kind)
        cclk.stop()
        configs["clocks"] = cclk.summary()
        w = w0
    else:
        w = work.w
    if rank == 0:
        cfg = workload_config(args.workload, w, world)
        cfg["rows_per_step"] = rows_per_step
        cfg["l2"] = l2
        line = {
            "metric": metric_of(w), "value": round(value, 1), "unit": UNIT,
            "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(ms_step, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": dtype_name(w),
            "data": "synthetic (seeded; shapes and distributions of the "
                    "pages' workloads)",
            "config": cfg,
            "tokens_per_s": round(tokens_per_step * steps * world
                                  / (ms / 1e3), 1),
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "parity": parity,
            "clocks": clocks.summary(),
            "gpu_launches": launches * steps,
            "configs": configs,
        }
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()


def dtype_name(w):
    import torch
    n = {torch.bfloat16: "bf16", torch.float32: "f32"}
    if w.temperature == 0:
        return n[w.target_dtype]
    return f"{n[w.target_dtype]}+{n[w.draft_dtype]} (f32 accumulate)"


# ------------------------------------------------------- KV-cache commit
# A 32-layer model's KV cache (K and V, 8 KV heads of 128 bf16 values),
# head-major [64, B, 8, S, 128], B = 32 sequences with 2048..4095 committed
# positions each; after verification of the 60-node static tree, each
# sequence keeps the path to a random node (none with probability 0.2).
# 64 seeded path sets cycle, so the rows a step touches are not left in L2
# by the previous steps (about 1.3 GB over the cycle).
KV = dict(L=32, H=8, D=128, B=32, N=60, pre_lo=2048, pre_hi=4096, sets=64)
KV_METRIC = "KV-cache commit bytes moved/s (read + write)"


def kv_paths(seed=11):
    """Path sets: prefix [P, B], length [P, B], nodes [P, B, N] (int32)."""
    import numpy as np
    import synth
    parent = synth.static_tree(synth.workload("tree_static")).numpy()
    N, B, P = KV["N"], KV["B"], KV["sets"]
    rng = np.random.default_rng(seed)
    pre = rng.integers(KV["pre_lo"], KV["pre_hi"], size=(P, B)).astype(np.int32)
    lens = np.zeros((P, B), dtype=np.int32)
    nodes = np.full((P, B, N), -1, dtype=np.int32)
    for k in range(P):
        for b in range(B):
            if rng.random() < 0.2:
                continue
            j, chain = int(rng.integers(0, N)), []
            while j >= 0:
                chain.append(j)
                j = int(parent[j])
            chain.reverse()
            lens[k, b] = len(chain)
            nodes[k, b, :len(chain)] = chain
    return pre, lens, nodes


def kv_moved_bytes(lens, nodes):
    """Bytes read + written per path set: 2 x row x planes per moved
    position (a path position already in place moves nothing)."""
    import numpy as np
    row = KV["D"] * 2 * 2 * KV["L"] * KV["H"]  # bf16 rows over all planes
    idx = np.arange(nodes.shape[-1])
    moved = ((nodes != idx) & (idx < lens[..., None])).sum(axis=-1)
    return moved.sum(axis=-1) * row * 2


def kv_oracle_rate(pre, lens, nodes, seconds):
    """The oracle on one sequence at a time (prefix cut to 64 positions so
    that the host copy of the cache stays small): bytes moved per second."""
    import numpy as np
    from oracle.kv import kv_commit
    N = KV["N"]
    cache = np.zeros((1, 64 + N, 2 * KV["L"] * KV["H"] * KV["D"]), np.int16)
    done, t0, i = 0, time.perf_counter(), 0
    P, B = lens.shape
    while True:
        k, b = (i // B) % P, i % B
        kv_commit(cache, [64], lens[k, b:b + 1], nodes[k, b:b + 1])
        done += int(kv_moved_bytes(lens[k, b:b + 1][None],
                                   nodes[k, b:b + 1][None])[0])
        i += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el / 1e9, i, el


def kv_main(args, world, rank, local):
    pre, lens, nodes = kv_paths()
    moved = kv_moved_bytes(lens, nodes)
    sample = ("sequences one by one through the oracle (numpy), prefix cut "
              "to 64 positions, {n} sequences in {el:.1f} s")
    if args.impl == "reference":
        if rank != 0:
            return
        steps = args.steps or 3
        for _ in range(args.warmup):
            kv_oracle_rate(pre, lens, nodes, 2.0)
        tot_b = tot_t = 0.0
        n_all = 0
        for _ in range(steps):
            r, n, el = kv_oracle_rate(pre, lens, nodes, 10.0)
            tot_b += r * el
            tot_t += el
            n_all += n
        v = tot_b / tot_t
        print(json.dumps({
            "impl": "reference", "metric": KV_METRIC, "value": round(v, 4),
            "unit": "GB/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(tot_t / steps * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 (bytes)", "data": "synthetic",
            "config": {"workload": "kv_commit", "B": KV["B"]},
            "cpu_baseline": {"kind": "oracle", "cores": 1, "value": round(v, 4),
                             "unit": "GB/s",
                             "sample": sample.format(n=n_all, el=tot_t)},
            "e2e": {"value": round(v, 4), "unit": "GB/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    import ctypes
    import torch
    import __graft_entry__ as g
    g.build()
    from speculative_decoding_verification_tree_gb300 import _lib, api
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    L2, H, D, B, N = 2 * KV["L"], KV["H"], KV["D"], KV["B"], KV["N"]
    S = KV["pre_hi"] + N
    cache = torch.zeros(L2, B, H, S, D, dtype=torch.bfloat16, device=dev)
    es = 2
    layout = (L2, H, H * S * D * es, B * H * S * D * es, S * D * es, D * es)
    d_pre = torch.tensor(pre, device=dev)
    d_len = torch.tensor(lens, device=dev)
    d_nodes = torch.tensor(nodes, device=dev)
    new_len = torch.empty(B, dtype=torch.int32, device=dev)
    P = KV["sets"]

    def step(k, ins=None):
        p_, l_, n_ = ins if ins is not None else (d_pre[k], d_len[k],
                                                   d_nodes[k])
        api.spec_kv_commit(cache, p_, l_, n_, layout=layout,
                           row_bytes=D * es, N=N, new_len=new_len)

    steps = args.steps or 3200
    warm = max(3, args.warmup)
    for k in range(warm):
        step(k % P)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    h = _lib.load()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    h.spec_profile_enable(PROFILE_EVERY)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for k in range(steps):
        step(k % P)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    tot, nl = ctypes.c_double(0), ctypes.c_int(0)
    rc = h.spec_profile_read(_lib.SPEC_PROF_KV, ctypes.byref(tot),
                             ctypes.byref(nl))
    h.spec_profile_enable(0)
    if ms < 1000.0 and not args.no_extend:
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for k in range(50):
                step(k % P)
            torch.cuda.synchronize()
    clocks.stop()
    ms = max_over_ranks(dist, ms, dev)
    bytes_run = float(sum(moved[k % P] for k in range(steps)))
    value = bytes_run * world / (ms / 1e3) / 1e9
    peak, peak_kind = _peaks()
    roof = None
    if nl.value:
        kern_ms = tot.value / nl.value
        per_launch = bytes_run / steps
        achieved = per_launch / (kern_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": None, "kernel": "kv_move",
                "bytes_per_launch": int(per_launch),
                "avg_launch_ms": round(kern_ms, 5), "peak_source": peak_kind,
                "profile_rc": rc}
    e2e = None
    if not args.no_e2e:
        h_pre = torch.tensor(pre).pin_memory()
        h_len = torch.tensor(lens).pin_memory()
        h_nodes = torch.tensor(nodes).pin_memory()
        h_out = torch.empty(B, dtype=torch.int32).pin_memory()
        x_pre = torch.empty(B, dtype=torch.int32, device=dev)
        x_len = torch.empty(B, dtype=torch.int32, device=dev)
        x_nodes = torch.empty(B, N, dtype=torch.int32, device=dev)
        n_e2e = 200

        def e2e_step(k):
            x_pre.copy_(h_pre[k], non_blocking=True)
            x_len.copy_(h_len[k], non_blocking=True)
            x_nodes.copy_(h_nodes[k], non_blocking=True)
            step(k, (x_pre, x_len, x_nodes))
            h_out.copy_(new_len, non_blocking=True)
        e2e_step(0)
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record()
        for k in range(n_e2e):
            e2e_step(k % P)
        a1.record()
        torch.cuda.synchronize()
        ems = max_over_ranks(dist, a0.elapsed_time(a1), dev)
        eb = float(sum(moved[k % P] for k in range(n_e2e)))
        e2e = {"value": round(eb * world / (ems / 1e3) / 1e9, 2),
               "unit": "GB/s", "h2d_bytes_per_step": B * (N + 2) * 4,
               "d2h_bytes_per_step": B * 4, "steps": n_e2e,
               "ms_per_step": round(ems / n_e2e, 4)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        r, n, el = kv_oracle_rate(pre, lens, nodes, min(args.cpu_seconds, 10))
        cpu = {"value": round(r, 4), "unit": "GB/s", "cores": 1,
               "kind": "oracle", "sample": sample.format(n=n, el=el)}
    if rank == 0:
        print(json.dumps({
            "metric": KV_METRIC, "value": round(value, 2), "unit": "GB/s",
            "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(ms / steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16 (bytes)",
            "data": "synthetic (seeded paths of the 60-node static tree)",
            "config": {"workload": "kv_commit", "B": B, "layers": KV["L"],
                       "kv_heads": H, "head_dim": D,
                       "layout": "head-major [2L, B, H, S, D]",
                       "positions": S, "path_sets": P,
                       "moved_positions_per_step": round(
                           float(moved.mean()) / (2 * D * es * L2 * H), 2),
                       "parallelism": f"replicas x{world} (sequences split)",
                       "l2": "64 path sets cycle over a "
                             f"{cache.numel() * es / 1e9:.1f} GB cache"},
            "roofline": roof, "cpu_baseline": cpu, "e2e": e2e,
            "clocks": clocks.summary(), "gpu_launches": 2 * steps}),
              flush=True)
    if dist:
        dist.destroy_process_group()


# ------------------------------------------------------ acceptance records
# The outcomes of verifying the 60-node static tree, B = 32 rounds per call
# (one verification step's batch; --B sets another): each round's path goes
# to a random node (none with probability 0.15), the drafter's confidence in
# each node's token is uniform on [0, 1], 20 confidence bins.  Seeded input
# sets cycle (64 at B = 32).
ST = dict(B=32, N=60, nbins=20, sets=64)
ST_METRIC = "verification rounds recorded/s (acceptance records)"


def stats_sets(B):
    """Input sets that cycle: 64 at the default batch, fewer for large
    batches (at least 4, and the cycle stays larger than L2)."""
    return max(4, min(ST["sets"], (1 << 20) // max(B, 1)))


def stats_inputs(B, seed=13):
    """count [P, B], parent [P, B, N], path [P, B, N] int32; conf [P, B, N]
    float32."""
    import numpy as np
    import synth
    tree = synth.static_tree(synth.workload("tree_static")).numpy()
    N, P = ST["N"], stats_sets(B)
    # root path of every node
    tab = np.full((N, N), -1, dtype=np.int32)
    tlen = np.zeros(N, dtype=np.int32)
    for j in range(N):
        chain, v = [], j
        while v >= 0:
            chain.append(v)
            v = int(tree[v])
        tab[j, :len(chain)] = chain[::-1]
        tlen[j] = len(chain)
    rng = np.random.default_rng(seed)
    target = rng.integers(0, N, size=(P, B))
    none = rng.random((P, B)) < 0.15
    count = np.where(none, 0, tlen[target]).astype(np.int32)
    path = np.where(none[..., None], -1, tab[target]).astype(np.int32)
    parent = np.ascontiguousarray(
        np.broadcast_to(tree, (P, B, N)).astype(np.int32))
    conf = rng.random((P, B, N)).astype(np.float32)
    return count, parent, path, conf


def stats_bytes(count, B):
    """Algorithmic bytes of one call: each round's count, parent row,
    confidence row and path prefix read once (records are < 1 KB)."""
    N = ST["N"]
    return B * (4 + 8 * N) + 4 * int(count.sum())


def stats_oracle_rate(count, parent, path, conf, seconds):
    from oracle.stats import accept_stats
    done, t0, k = 0, time.perf_counter(), 0
    P = count.shape[0]
    while True:
        accept_stats(count[k % P], parent[k % P], path[k % P], conf[k % P],
                     ST["N"], ST["nbins"])
        done += count.shape[1]
        k += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el, done, el


def stats_main(args, world, rank, local):
    B = args.B or ST["B"]
    count, parent, path, conf = stats_inputs(B)
    P, N, nb = count.shape[0], ST["N"], ST["nbins"]
    sample = "rounds through the oracle (numpy / Python), {n} rounds in {el:.1f} s"
    cfg = {"workload": "accept_stats", "B": B, "nodes": N, "nbins": nb,
           "tree": "60-node static tree (4,12,16,14,8,6)", "input_sets": P,
           "l2": f"{P} input sets cycle "
                 f"({P * stats_bytes(count[0], B) / 1e6:.1f} MB)"}
    if args.impl == "reference":
        if rank != 0:
            return
        steps = args.steps or 3
        for _ in range(args.warmup):
            stats_oracle_rate(count, parent, path, conf, 1.0)
        done = el = 0.0
        for _ in range(steps):
            _, d, e = stats_oracle_rate(count, parent, path, conf, 10.0)
            done += d
            el += e
        v = done / el
        print(json.dumps({
            "impl": "reference", "metric": ST_METRIC, "value": round(v, 1),
            "unit": "rounds/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int64 (counts) + f64 (sums)", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"kind": "oracle", "cores": 1, "value": round(v, 1),
                             "unit": "rounds/s",
                             "sample": sample.format(n=int(done), el=el)},
            "e2e": {"value": round(v, 1), "unit": "rounds/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    import ctypes
    import torch
    import __graft_entry__ as g
    g.build()
    from speculative_decoding_verification_tree_gb300 import _lib, api
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    d_count = torch.from_numpy(count).to(dev)
    d_parent = torch.from_numpy(parent).to(dev)
    d_path = torch.from_numpy(path).to(dev)
    d_conf = torch.from_numpy(conf).to(dev)
    rec = api.accept_stats_records(N, nb, dev)

    def step(k, ins=None):
        c, p_, q_, f_ = ins if ins is not None else (
            d_count[k], d_parent[k], d_path[k], d_conf[k])
        api.spec_accept_stats(c, p_, q_, f_, n=N, nbins=nb, out=rec)

    steps = args.steps or 2000
    warm = max(3, args.warmup)
    for k in range(warm):
        step(k % P)
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    h = _lib.load()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    h.spec_profile_enable(PROFILE_EVERY)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for k in range(steps):
        step(k % P)
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    tot, nl = ctypes.c_double(0), ctypes.c_int(0)
    rc = h.spec_profile_read(_lib.SPEC_PROF_STATS, ctypes.byref(tot),
                             ctypes.byref(nl))
    h.spec_profile_enable(0)
    if ms < 1000.0 and not args.no_extend:
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for k in range(50):
                step(k % P)
            torch.cuda.synchronize()
    clocks.stop()
    ms = max_over_ranks(dist, ms, dev)
    value = B * steps * world / (ms / 1e3)
    peak, peak_kind = _peaks()
    roof = None
    if nl.value:
        kern_ms = tot.value / nl.value
        per_launch = sum(stats_bytes(count[k % P], B)
                         for k in range(steps)) / steps
        achieved = per_launch / (kern_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 5),
                "traffic": _traffic("accept_stats", B),
                "kernel": "accept_stats_warp" if N <= 64 else
                          "accept_stats_cta",
                "bytes_per_launch": int(per_launch),
                "avg_launch_ms": round(kern_ms, 5), "peak_source": peak_kind,
                "profile_rc": rc}
    e2e = None
    if not args.no_e2e:
        h_in = [torch.from_numpy(a).pin_memory()
                for a in (count, parent, path, conf)]
        x_in = [torch.empty_like(a[0], device=dev) for a in h_in]
        h_out = {f: torch.empty_like(t, device="cpu").pin_memory()
                 for f, t in rec.items()}
        n_e2e = 500

        def e2e_step(k):
            for x, hh in zip(x_in, h_in):
                x.copy_(hh[k], non_blocking=True)
            step(k, x_in)
            for f, t in rec.items():
                h_out[f].copy_(t, non_blocking=True)
        e2e_step(0)
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record()
        for k in range(n_e2e):
            e2e_step(k % P)
        a1.record()
        torch.cuda.synchronize()
        ems = max_over_ranks(dist, a0.elapsed_time(a1), dev)
        e2e = {"value": round(B * n_e2e * world / (ems / 1e3), 1),
               "unit": "rounds/s",
               "h2d_bytes_per_step": sum(a[0].numel() * a.element_size()
                                         for a in h_in),
               "d2h_bytes_per_step": sum(t.numel() * t.element_size()
                                         for t in rec.values()),
               "steps": n_e2e, "ms_per_step": round(ems / n_e2e, 4)}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        r, n, el = stats_oracle_rate(count, parent, path, conf,
                                     min(args.cpu_seconds, 10))
        cpu = {"value": round(r, 1), "unit": "rounds/s", "cores": 1,
               "kind": "oracle", "sample": sample.format(n=n, el=el)}
    if rank == 0:
        cfg["parallelism"] = f"replicas x{world} (rounds split)"
        print(json.dumps({
            "metric": ST_METRIC, "value": round(value, 1), "unit": "rounds/s",
            "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(ms / steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "int32 in; int64 counts, f64 confidence sums",
            "data": "synthetic (seeded paths of the 60-node static tree)",
            "config": cfg, "roofline": roof, "cpu_baseline": cpu,
            "e2e": e2e, "clocks": clocks.summary(), "gpu_launches": steps}),
              flush=True)
    if dist:
        dist.destroy_process_group()


# ------------------------------------------------------------ tree attention
# One attention layer of the verification pass of a Llama-3-8B-shaped target
# (32 query heads over 8 key/value heads, head dim 128, bf16): B = 32
# sequences with committed prefixes of 2048..4095 positions, the 60-node
# static tree drafted after each.  The caches (2 x 272 MB) exceed L2.
AT = dict(B=32, Hq=32, Hkv=8, D=128, pre_lo=2048, pre_hi=4096)
AT_METRIC = "tree-attention verified draft tokens/s (one layer)"


def attn_inputs(B, seed=31):
    import numpy as np
    import synth
    tree = synth.static_tree(synth.workload("tree_static")).numpy()
    rng = np.random.default_rng(seed)
    prefix = rng.integers(AT["pre_lo"], AT["pre_hi"], size=B).astype(np.int32)
    return tree, prefix


def attn_work(prefix, N):
    """Algorithmic bytes (each key / value row of the range once, q, out)
    and FLOPs (QK and PV over every key of the range) of one call."""
    H, Hq, D = AT["Hkv"], AT["Hq"], AT["D"]
    keys = int(prefix.sum()) + len(prefix) * N
    nbytes = keys * H * D * 2 * 2 + 2 * len(prefix) * N * Hq * D * 2
    flops = 4 * keys * N * Hq * D
    return nbytes, flops


def attn_oracle_rate(tree, prefix, seconds):
    """The oracle on one sequence at a time (prefix cut to 256 positions so
    that a sample finishes): draft tokens per second."""
    import numpy as np
    from oracle.attention import tree_attention
    rng = np.random.default_rng(0)
    N, Hq, H, D = tree.size, AT["Hq"], AT["Hkv"], AT["D"]
    P = 256
    q = rng.normal(size=(1, N, Hq, D))
    k = rng.normal(size=(1, H, P + N, D))
    v = rng.normal(size=(1, H, P + N, D))
    done, t0 = 0, time.perf_counter()
    while True:
        tree_attention(q, k, v, [P], tree[None], D ** -0.5)
        done += N
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el, done, el


def attn_device_inputs(torch, tree, prefix, dev):
    """q, the K / V caches, prefix lengths, mask rows (this library's
    spec_tree_mask of the tree) and the output of the tree-attention
    workload on the device (seeded)."""
    import numpy as np
    from speculative_decoding_verification_tree_gb300 import api
    B, N = len(prefix), tree.size
    Hq, H, D = AT["Hq"], AT["Hkv"], AT["D"]
    S = AT["pre_hi"] + 64
    gen = torch.Generator(device=dev)
    gen.manual_seed(37)
    q = torch.randn(B, N, Hq, D, generator=gen, device=dev).bfloat16()
    kc = torch.randn(B, H, S, D, generator=gen, device=dev).bfloat16()
    vc = torch.randn(B, H, S, D, generator=gen, device=dev).bfloat16()
    parent = torch.from_numpy(np.tile(tree, (B, 1)).astype(np.int32)).to(dev)
    _, bits = api.spec_tree_mask(parent, bits=True, mask=False)
    pre = torch.from_numpy(prefix).to(dev)
    return q, kc, vc, pre, bits, torch.empty_like(q)


def attn_roofline(prefix, N, kern_ms, peak):
    """HBM and tensor fractions of one tree-attention launch."""
    nbytes, flops = attn_work(prefix, N)
    achieved = nbytes / (kern_ms / 1e3) / 1e9
    tf = flops / (kern_ms / 1e3) / 1e12
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            tpk = float(json.load(f)["bf16_tflops"])
    except (OSError, KeyError, ValueError):
        tpk = 1900.0
    return nbytes, flops, achieved, tf, tpk


def attn_config(torch, h, lib, dev, steps, peak, peak_kind):
    """The tree-attention workload (B = 32, the static tree) timed inside
    the default run: launch time and its HBM and tensor fractions."""
    from speculative_decoding_verification_tree_gb300 import api
    tree, prefix = attn_inputs(AT["B"])
    q, kc, vc, pre, bits, out = attn_device_inputs(torch, tree, prefix, dev)
    for _ in range(5):
        api.spec_tree_attention(q, kc, vc, pre, bits, out=out)
    torch.cuda.synchronize()
    h.spec_profile_enable(PROFILE_EVERY)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        api.spec_tree_attention(q, kc, vc, pre, bits, out=out)
    e1.record()
    torch.cuda.synchronize()
    kern_ms, nl, rc = kernel_time(h, lib.SPEC_PROF_ATTN)
    h.spec_profile_enable(0)
    ms = e0.elapsed_time(e1)
    N = tree.size
    d = {"metric": AT_METRIC, "unit": "tokens/s",
         "value": round(AT["B"] * N * steps / (ms / 1e3), 1),
         "ms_per_step": round(ms / steps, 5), "steps": steps,
         "B": AT["B"], "nodes": N, "q_heads": AT["Hq"], "kv_heads": AT["Hkv"],
         "head_dim": AT["D"], "prefix": f"{AT['pre_lo']}..{AT['pre_hi'] - 1}",
         "dtype": "bf16 (f32 softmax and accumulation)",
         "l2": "K and V caches (2 x 272 MB) exceed L2",
         "kernel": "tree_attn_tc", "profile_rc": rc, "gpu_launches": steps,
         "avg_launch_ms": None if kern_ms is None else round(kern_ms, 5)}
    if kern_ms:
        nbytes, flops, achieved, tf, tpk = attn_roofline(prefix, N, kern_ms, peak)
        d.update({"bytes_per_launch": int(nbytes), "achieved_gbs": round(achieved, 1),
                  "peak_gbs": peak, "peak_source": peak_kind,
                  "frac": round(achieved / peak, 4),
                  "tensor": {"achieved_tflops": round(tf, 1), "peak_tflops": tpk,
                             "frac": round(tf / tpk, 4),
                             "flops_per_launch": int(flops)}})
    del q, kc, vc, pre, bits, out
    torch.cuda.empty_cache()
    return d


def attn_main(args, world, rank, local):
    B = args.B or AT["B"]
    tree, prefix = attn_inputs(B)
    N = tree.size
    sample = ("sequences of the oracle (numpy float64) with the prefix cut to "
              "256 positions, {n} draft tokens in {el:.1f} s")
    cfg = {"workload": "tree_attention", "B": B, "nodes": N, "q_heads": AT["Hq"],
           "kv_heads": AT["Hkv"], "head_dim": AT["D"],
           "prefix": f"{AT['pre_lo']}..{AT['pre_hi'] - 1}",
           "tree": "60-node static tree (4,12,16,14,8,6)",
           "l2": "K and V caches (2 x 272 MB at B=32) exceed L2"}
    if args.impl == "reference":
        if rank != 0:
            return
        steps = args.steps or 3
        for _ in range(args.warmup):
            attn_oracle_rate(tree, prefix, 1.0)
        done = el = 0.0
        for _ in range(steps):
            _, d, e = attn_oracle_rate(tree, prefix, 10.0)
            done += d
            el += e
        v = done / el
        print(json.dumps({
            "impl": "reference", "metric": AT_METRIC, "value": round(v, 2),
            "unit": "tokens/s", "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 1),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"kind": "oracle", "cores": 1, "value": round(v, 2),
                             "unit": "tokens/s",
                             "sample": sample.format(n=int(done), el=el)},
            "e2e": {"value": round(v, 2), "unit": "tokens/s",
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}),
              flush=True)
        return
    import ctypes
    import numpy as np
    import torch
    import __graft_entry__ as g
    g.build()
    from speculative_decoding_verification_tree_gb300 import _lib, api
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    q, kc, vc, pre, bits, out = attn_device_inputs(torch, tree, prefix, dev)

    def step(ins=None):
        q_, p_, b_ = ins if ins is not None else (q, pre, bits)
        api.spec_tree_attention(q_, kc, vc, p_, b_, out=out)

    steps = args.steps or 300
    warm = max(3, args.warmup)
    for _ in range(warm):
        step()
    torch.cuda.synchronize()
    clocks = Clocks(local)
    clocks.start()
    time.sleep(0.3)
    h = _lib.load()
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    h.spec_profile_enable(PROFILE_EVERY)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(steps):
        step()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1)
    tot, nl = ctypes.c_double(0), ctypes.c_int(0)
    rc = h.spec_profile_read(_lib.SPEC_PROF_ATTN, ctypes.byref(tot),
                             ctypes.byref(nl))
    h.spec_profile_enable(0)
    if ms < 1000.0 and not args.no_extend:
        t_end = time.time() + 1.0
        while time.time() < t_end:
            for _ in range(20):
                step()
            torch.cuda.synchronize()
    clocks.stop()
    ms = max_over_ranks(dist, ms, dev)
    value = B * N * steps * world / (ms / 1e3)
    nbytes, flops = attn_work(prefix, N)
    peak, peak_kind = _peaks()
    roof = None
    if nl.value:
        kern_ms = tot.value / nl.value
        nbytes, flops, achieved, tf, tpk = attn_roofline(prefix, N, kern_ms,
                                                         peak)
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                "unit": "GB/s", "frac": round(achieved / peak, 4),
                "traffic": None, "kernel": "tree_attn_tc",
                "bytes_per_launch": int(nbytes),
                "avg_launch_ms": round(kern_ms, 5), "peak_source": peak_kind,
                "tensor": {"achieved_tflops": round(tf, 1),
                           "peak_tflops": tpk, "frac": round(tf / tpk, 4),
                           "flops_per_launch": int(flops),
                           "path": "tcgen05.mma kind::f16, TMEM "
                                   "accumulators, K/V by TMA"},
                "profile_rc": rc}
    e2e = None
    if not args.no_e2e:
        h_q = q.cpu().pin_memory()
        h_pre = pre.cpu().pin_memory()
        h_bits = bits.cpu().pin_memory()
        h_out = torch.empty_like(out, device="cpu").pin_memory()
        x_q, x_pre, x_bits = (torch.empty_like(q), torch.empty_like(pre),
                              torch.empty_like(bits))
        n_e2e = 100

        def e2e_step():
            x_q.copy_(h_q, non_blocking=True)
            x_pre.copy_(h_pre, non_blocking=True)
            x_bits.copy_(h_bits, non_blocking=True)
            step((x_q, x_pre, x_bits))
            h_out.copy_(out, non_blocking=True)
        e2e_step()
        torch.cuda.synchronize()
        a0 = torch.cuda.Event(enable_timing=True)
        a1 = torch.cuda.Event(enable_timing=True)
        a0.record()
        for _ in range(n_e2e):
            e2e_step()
        a1.record()
        torch.cuda.synchronize()
        ems = max_over_ranks(dist, a0.elapsed_time(a1), dev)
        e2e = {"value": round(B * N * n_e2e * world / (ems / 1e3), 1),
               "unit": "tokens/s",
               "h2d_bytes_per_step": q.numel() * 2 + B * 4 + B * N * 8,
               "d2h_bytes_per_step": out.numel() * 2,
               "steps": n_e2e, "ms_per_step": round(ems / n_e2e, 4),
               "note": "the K/V caches stay resident (they are the model's "
                       "state, not a per-step input)"}
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        r, n, el = attn_oracle_rate(tree, prefix, min(args.cpu_seconds, 10))
        cpu = {"value": round(r, 2), "unit": "tokens/s", "cores": 1,
               "kind": "oracle", "sample": sample.format(n=n, el=el)}
    if rank == 0:
        cfg["parallelism"] = f"replicas x{world} (sequences split)"
        print(json.dumps({
            "metric": AT_METRIC, "value": round(value, 1), "unit": "tokens/s",
            "n_gpus": world, "steps": steps, "warmup": warm,
            "ms_per_step": round(ms / steps, 5), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16 (f32 softmax and accumulation)",
            "data": "synthetic (seeded N(0,1) q, k, v; static tree)",
            "config": cfg, "roofline": roof, "cpu_baseline": cpu,
            "e2e": e2e, "clocks": clocks.summary(), "gpu_launches": steps}),
              flush=True)
    if dist:
        dist.destroy_process_group()


def reference_arm(args, world, rank):
    if rank != 0:
        return
    steps = args.steps or 3
    w, host = host_inputs(args.workload)
    per_step = max(0.2, min(args.cpu_seconds, 150.0 / (steps + args.warmup)))
    for _ in range(args.warmup):
        time_oracle(args.workload, per_step, (w, host))
    rows, el = 0, 0.0
    nseq = 0
    for _ in range(steps):
        r, n, e = time_oracle(args.workload, per_step, (w, host))
        rows += r * e
        el += e
        nseq += n
    value = rows / el
    import synth
    wf = synth.workload(args.workload)  # the workload our arm times
    line = {"impl": "reference", "metric": metric_of(wf),
            "value": round(value, 2),
            "unit": UNIT, "n_gpus": world, "steps": steps,
            "warmup": args.warmup, "ms_per_step": round(el / steps * 1e3, 2),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, wf, world),
            "cpu_baseline": {"kind": "oracle", "cores": 1,
                             "sample": cpu_sample_text(args.workload, nseq,
                                                       el),
                             "value": round(value, 2), "unit": UNIT},
            "e2e": {"value": round(value, 2), "unit": UNIT,
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

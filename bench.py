#!/usr/bin/env python
"""Throughput of the packed-sequence preprocessing hot path on GB300.

One step is one pass of the whole hot path over one batch of each of the
five synthetic workloads (all inputs resident in HBM when timing starts):

  map_small   pseq_from_doc_ids on doc_ids int32 [4, 2048]
  thd_small   thd_from_batch of the matching int64 ids / labels / positions
  thd_ids     thd_from_batch, B=8 S=8192, 64 pack slots, int64 ids, labels,
              mRoPE positions [3, 8, 8192]
  thd_emb     thd_from_batch of bf16 hidden [4, 8192, 4096]
  squeeze     pack_squeeze of int64 [256, 4096] into FFD bins of 32768
  map_stress  pseq_from_doc_ids on doc_ids int32 [64, 32768] (~250k segments)

Metric: packed tokens per second (tokens of every produced stream: B*S per
map, T per THD stream, bins*width per squeeze) and achieved HBM GB/s of the
dominant kernel (the embedding gather) against the measured copy bandwidth.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
For N > 1 launch under torchrun; every rank runs its own batches (weak
scaling, no data-path collective) and rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "packed tokens/sec and achieved HBM GB/s (% of GB300 peak), 1 GPU"
EMB_SAMPLE = 2  # the embedding call's end is marked with an event on every 2nd timed step
UNIT = "tokens/s"
L2_FLUSH_BYTES = 256 << 20
WORKLOAD = ("packed-sequence preprocessing step: doc_ids map [4,2048] + its THD batch (int64 ids/labels/positions); "
            "THD B=8 S=8192 64 packs (ids, labels, mRoPE [3,8,8192]); THD bf16 hidden [4,8192,4096]; "
            "squeeze int64 [256,4096] -> FFD bins x 32768; doc_ids map [64,32768] (~250k segments)")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--profile-calls", action="store_true",
                    help="issue every configuration's call (and the scaled squeeze and next-row calls) a few "
                         "times, untimed, for a profiler to capture; prints no JSON line")
    return ap.parse_args()


# ----------------------------------------------------------------------------
# distributed plumbing (timing only; the path itself exchanges nothing)
# ----------------------------------------------------------------------------
class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None

    def init(self, backend: str):
        if self.world > 1:
            import torch.distributed as dist

            dist.init_process_group(backend=backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float, device=None) -> float:
        if self.pg is None:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def sum(self, x: float, device=None) -> float:
        if self.pg is None:
            return x
        import torch

        t = torch.tensor([x], dtype=torch.float64, device=device)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.SUM)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ----------------------------------------------------------------------------
# inputs
# ----------------------------------------------------------------------------
def make_inputs(seed: int) -> dict:
    """Host inputs of every part of one step (numpy; hidden as torch bf16)."""
    small = synth.doc_map_small(seed)
    return {
        "map_small": small["doc_ids"],
        "thd_small": {k: small[k] for k in ("input_ids", "labels", "position_ids", "seq_lens", "seq_lens_padded")},
        "thd_ids": synth.thd_ids(seed),
        "thd_emb": synth.thd_embeddings(seed),
        "squeeze": synth.squeeze(seed),
        "map_stress": synth.doc_map_stress(seed),
    }


# fields each id-stream THD part moves (name, planes); int64 elements, one per token
THD_FIELDS = {
    "thd_small": (("input_ids", 1), ("labels", 1), ("position_ids", 1)),
    "thd_ids": (("input_ids", 1), ("labels", 1), ("position_ids", 3)),
}
L2_NOTE = "flushed between steps outside the timed events (256 MiB write, then 256 MiB read of another buffer)"


def part_bytes(name: str, part, count: int, total: int) -> int:
    """Algorithmic bytes of one call -- what the method must read and write --
    from the call's inputs and what it produced: ``count`` segments, kept
    sequences or bin members, ``total`` tokens in the produced stream."""
    if name.startswith("map"):
        return part.size * 4 + 4 * (count + 1)
    if name.startswith("thd"):
        if "hidden" in part:
            moved = 2 * total * part["hidden"].shape[2] * 2
        else:
            moved = sum(2 * planes * total * 8 for _, planes in THD_FIELDS[name])
        return moved + total + 8 * (count + 1) + 2 * 8 * part["seq_lens"].size
    nb = len(part["bin_offsets"]) - 1
    return 8 * int(part["real_lens"].sum()) + 9 * nb * part["width"] + 8 * (count + nb)


def step_config(tokens: dict, alg_bytes: dict, world: int) -> dict:
    """The ``config`` of the JSON line, the same for both arms: the workload,
    its tokens and algorithmic bytes per step, how L2 is handled."""
    return {
        "workload": WORKLOAD,
        "tokens_per_step_per_gpu": int(sum(tokens.values())),
        "parts_tokens": {k: int(tokens[k]) for k in sorted(tokens)},
        "algorithmic_bytes_per_step": int(sum(alg_bytes.values())),
        "l2": L2_NOTE,
        "parallelism": f"replicas x{world} (independent batches per GPU)",
    }


# ----------------------------------------------------------------------------
# native arm
# ----------------------------------------------------------------------------
class NativeStep:
    """Device buffers and the C ABI calls of one step.

    Every call's ctypes arguments are built once, so issuing a step costs a
    handful of microseconds of CPU time; nothing is allocated per step.  All
    calls go to ``stream``.  ``host_pinned`` (shared between instances) holds
    the pinned host copy of every input for the end-to-end leg.
    """

    def __init__(self, host: dict, device, stream, host_pinned=None, side_stream=None, only=None):
        import torch

        import varlen_attention_metadata_gb300 as v

        self.torch = torch
        self.v = v
        self.lib = v.load_library()
        self.dev = device
        self.stream = stream
        self.sh = ctypes.c_void_p(stream.cuda_stream)
        # the embedding conversion may run on its own stream, next to the rest
        self.side = side_stream
        self.side_sh = ctypes.c_void_p(side_stream.cuda_stream) if side_stream is not None else self.sh
        self.host = host
        self.pinned = host_pinned if host_pinned is not None else {}
        self.inputs = []   # (device tensor, pinned host tensor) copied in by the end-to-end leg
        self.outputs = []  # (device tensor, nbytes) copied out by the end-to-end leg
        self.tokens = {}
        self.alg_bytes = {}
        self.calls = []    # (name, C function, argument tuple)
        self._finish = {}
        self._keep = []
        self._fork = self.torch.cuda.Event()
        self._join = self.torch.cuda.Event()
        self.only = set(only) if only else None
        self._build()

    def _in(self, key, a):
        torch = self.torch
        if key not in self.pinned:
            t = a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))
            self.pinned[key] = t.contiguous().pin_memory()
        h = self.pinned[key]
        d = torch.empty(h.shape, dtype=h.dtype, device=self.dev)
        d.copy_(h)
        self.inputs.append((d, h))
        return d

    def _zeros(self, n, dtype):
        return self.torch.zeros(n, dtype=dtype, device=self.dev)

    @staticmethod
    def _p(t, off=0):
        return ctypes.c_void_p(t.data_ptr() + off)

    def _map(self, name, doc_ids):
        torch, lib = self.torch, self.lib
        B, S = doc_ids.shape
        d = self._in(name, doc_ids)
        cu = self._zeros(B * S + 1, torch.int32)
        info = self._zeros(8, torch.int32)
        ws = self._zeros(lib.pseq_from_doc_ids_workspace_size(B, S), torch.uint8)
        args = (self._p(d), 4, B, S, self._p(cu), self._p(info), self._p(ws), ws.numel(), self.sh)
        self.calls.append((name, lib.pseq_from_doc_ids, args))
        self.tokens[name] = B * S
        self._keep.append((d, cu, info, ws))
        self._finish[name] = lambda: (info, cu, d)

    def _thd(self, name, batch, fields_np, hidden=None):
        torch, lib, v = self.torch, self.lib, self.v
        real, padded = batch["seq_lens"], batch["seq_lens_padded"]
        B, P = real.shape
        S = (fields_np[0][1] if fields_np else hidden).shape[1]
        dreal, dpad = self._in(name + ".seq_lens", real), self._in(name + ".seq_lens_padded", padded)
        fields = (v._lib.PseqField * 8)()
        dsts, srcs = [], []
        k = 0
        for fname, a, planes in fields_np:
            src = self._in(name + "." + fname, a)
            row = int(np.prod(a.shape[3 if planes > 1 else 2:])) if a.ndim > (3 if planes > 1 else 2) else 1
            dst = self._zeros(planes * B * S * row, src.dtype)
            fields[k].src, fields[k].dst = src.data_ptr(), dst.data_ptr()
            fields[k].elem_bytes, fields[k].planes, fields[k].row_elems = src.element_size(), planes, row
            dsts.append((dst, planes, row, src.element_size()))
            srcs.append(src)
            k += 1
        if hidden is not None:
            src = self._in(name + ".hidden", hidden)
            H = hidden.shape[2]
            dst = self._zeros(B * S * H, src.dtype)
            fields[k].src, fields[k].dst = src.data_ptr(), dst.data_ptr()
            fields[k].elem_bytes, fields[k].planes, fields[k].row_elems = 2, 1, H
            dsts.append((dst, 1, H, 2))
            srcs.append(src)
            k += 1
        cu = self._zeros(B * P + 1, torch.int32)
        cup = self._zeros(B * P + 1, torch.int32)
        mask = self._zeros(B * S, torch.uint8)
        info = self._zeros(8, torch.int32)
        ws = self._zeros(lib.thd_workspace_size(B, P), torch.uint8)
        self._keep.append((fields, srcs, dreal, dpad, cu, cup, mask, info, ws))
        args = (self._p(dreal), self._p(dpad), B, S, P, -1000, 1, fields, k, self._p(cu), self._p(cup),
                self._p(mask), self._p(info, 16), self._p(info), self._p(ws), ws.numel(), self.sh)
        self.calls.append((name, lib.thd_from_batch, args))
        self._finish[name] = lambda: (info, cu, cup, mask, dsts)

    def _squeeze(self, name, c):
        torch, lib = self.torch, self.lib
        src = self._in(name + ".src", c["src"])
        real = self._in(name + ".real_lens", c["real_lens"])
        offs = self._in(name + ".bin_offsets", c["bin_offsets"])
        mem = self._in(name + ".bin_members", c["bin_members"])
        N, W = c["src"].shape
        nb, M = len(c["bin_offsets"]) - 1, int(c["bin_offsets"][-1])
        width = c["width"]
        out = self._zeros(nb * width, torch.int64)
        mask = self._zeros(nb * width, torch.uint8)
        cu = self._zeros(M + nb + 1, torch.int32)
        cup = self._zeros(M + nb + 1, torch.int32)
        info = self._zeros(8, torch.int32)
        ws = self._zeros(lib.pack_squeeze_workspace_size(M, nb), torch.uint8)
        self._keep.append((src, real, offs, mem, out, mask, cu, cup, info, ws))
        args = (self._p(src), N, W, 8, self._p(real), self._p(offs), self._p(mem), nb, M, c["multiple"],
                c["capacity"], 1 if c["stretch"] else 0, width, c["pad_value"], self._p(out), self._p(cu),
                self._p(cup), self._p(mask), self._p(info), self._p(ws), ws.numel(), self.sh)
        self.calls.append((name, lib.pack_squeeze, args))
        self.tokens[name] = nb * width
        self._finish[name] = lambda: (info, cu, cup, mask, out, M + nb)

    def _want(self, name):
        return name in self.host and (self.only is None or name in self.only)

    def _build(self):
        h = self.host
        if self._want("map_small"):
            self._map("map_small", h["map_small"])
        if self._want("thd_small"):
            t0 = h["thd_small"]
            self._thd("thd_small", t0, [("input_ids", t0["input_ids"], 1), ("labels", t0["labels"], 1),
                                        ("position_ids", t0["position_ids"], 1)])
        if self._want("thd_ids"):
            t1 = h["thd_ids"]
            self._thd("thd_ids", t1, [("input_ids", t1["input_ids"], 1), ("labels", t1["labels"], 1),
                                      ("position_ids", t1["position_ids"], 3)])
        if self._want("thd_emb"):
            self._thd("thd_emb", h["thd_emb"], [], hidden=h["thd_emb"]["hidden"])
        if self._want("squeeze"):
            self._squeeze("squeeze", h["squeeze"])
        if self._want("map_stress"):
            self._map("map_stress", h["map_stress"])
        # extras timed on their own only (never part of the step): a larger
        # squeeze, and the embedding batch with rows that end short
        if self.only is not None and self._want("squeeze_scaled"):
            self._squeeze("squeeze_scaled", h["squeeze_scaled"])
        if self.only is not None and self._want("thd_emb_ragged"):
            self._thd("thd_emb_ragged", h["thd_emb_ragged"], [], hidden=h["thd_emb_ragged"]["hidden"])
        # the same calls with the side stream's handle (every ABI call takes its stream last)
        self.side_calls = [(name, fn, args[:-1] + (self.side_sh,)) for name, fn, args in self.calls]
        self.torch.cuda.synchronize(self.dev)

    def run(self, emb_end=None, two_streams=False):
        """Issue one step; optionally mark the end of the embedding call with
        an event (it is the step's first call, so the step's start event
        marks its start).

        The embedding conversion goes first, on self.stream.  With two_streams
        the other calls go to the side stream (forked from and joined back
        into self.stream), so they run next to it while it streams its
        537 MB: issued first, with no cross-stream wait in front of it, the
        embedding call's CTAs take their SMs before the small calls' CTAs
        arrive, and the small calls fill the SMs it leaves free."""
        two = two_streams and self.side is not None
        if two:
            self._fork.record(self.stream)
            self.side.wait_event(self._fork)
        for name, fn, args in self.calls:
            if name != "thd_emb":
                continue
            self._ok(name, fn(*args))
            if emb_end is not None:
                emb_end.record(self.stream)
        for name, fn, args in (self.side_calls if two else self.calls):
            if name != "thd_emb":
                self._ok(name, fn(*args))
        if two:
            self._join.record(self.side)
            self.stream.wait_event(self._join)

    def _ok(self, name, status):
        # a call that enqueued nothing must not pass for a fast one
        if status != 0:
            raise RuntimeError(f"{name}: status {status}: {self.v.load_library().pseq_last_error().decode()}")

    def resolve(self):
        """After one untimed step: exact token counts, output sizes, checks."""
        torch = self.torch
        torch.cuda.synchronize(self.dev)
        self.outputs = []
        for name, get in self._finish.items():
            res = get()
            info = res[0][:4].tolist()
            if info[0] != 0:
                raise RuntimeError(f"{name}: device status {info[0]}")
            if name.startswith("map"):
                _, cu, d = res
                self.outputs.append((cu, 4 * (info[1] + 1)))
            elif name.startswith("thd"):
                _, cu, cup, mask, dsts = res
                n, T = info[1], info[3]
                self.tokens[name] = T
                self.outputs += [(cu, 4 * (n + 1)), (cup, 4 * (n + 1)), (mask, T)]
                for dst, planes, row, eb in dsts:
                    self.outputs.append((dst, planes * T * row * eb))
            else:
                _, cu, cup, mask, out, ncu = res
                self.outputs += [(cu, 4 * ncu), (cup, 4 * ncu), (mask, mask.numel()), (out, out.numel() * 8)]
            self.alg_bytes[name] = part_bytes(name, self.host[name], info[1], info[3])
        self.emb_bytes = self.alg_bytes.get("thd_emb")
        self.h2d_bytes = sum(h.numel() * h.element_size() for _, h in self.inputs)
        self.d2h_bytes = sum(n for _, n in self.outputs)
        self.host_out = [torch.empty(n, dtype=torch.uint8, pin_memory=True) for _, n in self.outputs]

    def copy_in(self):
        for d, h in self.inputs:
            d.copy_(h, non_blocking=True)

    def copy_out(self):
        for (d, n), h in zip(self.outputs, self.host_out):
            h.copy_(d.view(self.torch.uint8)[:n], non_blocking=True)


def time_next_rows(dev, stream, seed: int, flush_l2, reps: int = 60) -> dict:
    """Per-call device time of the entry points beyond the step, each on a
    workload of the same family (event-timed medians, L2 flushed before every
    call, prebuilt ctypes arguments)."""
    import torch

    import varlen_attention_metadata_gb300 as v

    lib = v.load_library()
    P = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)  # noqa: E731
    sh = ctypes.c_void_p(stream.cuda_stream)
    keep = []

    def dev_t(a):
        t = torch.from_numpy(np.ascontiguousarray(a)).to(dev)
        keep.append(t)
        return t

    graph_us = {}

    def timed(fn, args):
        ts = []
        with torch.cuda.stream(stream):
            for i in range(reps + 5):
                flush_l2()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                st = fn(*args)
                b.record(stream)
                if st != 0:
                    raise RuntimeError(f"next-row call: status {st}")
                ts.append((a, b))
        torch.cuda.synchronize(dev)
        # back-to-back calls replayed from one CUDA graph: launch gaps removed
        graph_us[id(fn)] = _graph_us([(fn, args)] * 20, dev, stream, flush_l2) / 20 if reps > 1 else None
        return statistics.median(x.elapsed_time(y) * 1e3 for x, y in ts[5:])

    def g(fn):
        v = graph_us.get(id(fn))
        return round(v, 2) if v is not None else None

    out = {}
    # split_batch_into_thd_chunks: the B=8 S=8192 batch as 4 chunks of 2 rows
    c1 = synth.thd_ids(seed)
    B, S = c1["input_ids"].shape
    Pk = c1["seq_lens"].shape[1]
    fields = (v._lib.PseqField * 3)()
    dsts = []
    for k, (a, planes) in enumerate(((c1["input_ids"], 1), (c1["labels"], 1), (c1["position_ids"], 3))):
        src = dev_t(a)
        dst = torch.empty(planes * B * S, dtype=torch.int64, device=dev)
        keep.append(dst)
        fields[k].src, fields[k].dst, fields[k].elem_bytes, fields[k].planes, fields[k].row_elems = \
            src.data_ptr(), dst.data_ptr(), 8, planes, 1
    nc = 4
    real, pad = dev_t(c1["seq_lens"]), dev_t(c1["seq_lens_padded"])
    cu = torch.empty(nc * (B // nc * Pk + 1), dtype=torch.int32, device=dev)
    cup = torch.empty_like(cu)
    mask = torch.empty(B * S, dtype=torch.uint8, device=dev)
    infos = torch.empty(nc * 4, dtype=torch.int32, device=dev)
    pbs = torch.empty(nc, dtype=torch.uint8, device=dev)
    ws = torch.empty(lib.thd_workspace_size(B // nc, Pk), dtype=torch.uint8, device=dev)
    keep += [cu, cup, mask, infos, pbs, ws]
    us = timed(lib.thd_chunks_from_batch, (P(real), P(pad), B, S, Pk, nc, -1000, 1, fields, 3, P(cu), P(cup), P(mask),
                                           P(pbs), P(infos), P(ws), ws.numel(), sh))
    T = int(infos.view(nc, 4)[:, 3].sum().item())
    nbytes = 2 * T * 5 * 8 + T + 16 * B * Pk
    out["split_batch_into_thd_chunks"] = {"workload": "B=8 S=8192 ids/labels/mRoPE, 4 chunks", "us": round(us, 2),
                                          "graph_us": g(lib.thd_chunks_from_batch), "bytes": nbytes,
                                          "gbs": round(nbytes / us / 1e3, 1)}
    # thd_padding_mask (the standalone a8 call): the B=8 S=8192 batch's kept lengths
    kept = c1["seq_lens"] != -1000
    vr, vp = dev_t(c1["seq_lens"][kept]), dev_t(c1["seq_lens_padded"][kept])
    nk = int(kept.sum())
    Tk = int(c1["seq_lens_padded"][kept].sum())
    pmask = torch.empty(Tk, dtype=torch.uint8, device=dev)
    pinfo = torch.empty(4, dtype=torch.int32, device=dev)
    pws = torch.empty(lib.thd_workspace_size(1, nk), dtype=torch.uint8, device=dev)
    keep += [pmask, pinfo, pws]
    us = timed(lib.thd_padding_mask, (Tk, P(vr), P(vp), nk, P(pmask), P(pinfo), P(pws), pws.numel(), sh))
    nbytes = Tk + 16 * nk
    out["thd_padding_mask"] = {"workload": f"{nk} kept sequences of the B=8 S=8192 batch -> mask [{Tk}]",
                               "us": round(us, 2), "graph_us": g(lib.thd_padding_mask), "bytes": nbytes,
                               "gbs": round(nbytes / us / 1e3, 1)}
    # thd_padding_mask_from_token_ids: a 2M-token id stream with a padded tail
    rng = np.random.default_rng(seed)
    n = 1 << 21
    ids_np = rng.integers(1, 32000, size=n).astype(np.int64)
    ids_np[n - 4096:] = 0
    ids = dev_t(ids_np)
    tmask = torch.empty(n, dtype=torch.uint8, device=dev)
    tinfo = torch.empty(4, dtype=torch.int32, device=dev)
    tws = torch.zeros(lib.thd_mask_from_token_ids_workspace_size(n), dtype=torch.uint8, device=dev)
    keep += [tmask, tinfo, tws]
    us = timed(lib.thd_mask_from_token_ids, (P(ids), 8, n, 0, P(tmask), P(tinfo), P(tws), tws.numel(), sh))
    nbytes = 9 * n
    out["thd_padding_mask_from_token_ids"] = {"workload": "int64 ids [2097152], 4096-token pad tail",
                                              "us": round(us, 2), "graph_us": g(lib.thd_mask_from_token_ids),
                                              "bytes": nbytes, "gbs": round(nbytes / us / 1e3, 1)}
    # first-fit-decreasing: the squeeze workload's 256 lengths at capacity 32768
    c3 = synth.squeeze(seed)
    lens = dev_t(c3["real_lens"])
    offs = torch.empty(len(c3["real_lens"]) + 1, dtype=torch.int32, device=dev)
    mem = torch.empty(len(c3["real_lens"]), dtype=torch.int32, device=dev)
    finfo = torch.empty(4, dtype=torch.int32, device=dev)
    keep += [offs, mem, finfo]
    us = timed(lib.pack_ffd, (P(lens), len(c3["real_lens"]), c3["multiple"], c3["capacity"], P(offs), P(mem),
                              P(finfo), sh))
    out["first_fit_decreasing"] = {"workload": "256 lengths, multiple 64, capacity 32768", "us": round(us, 2),
                                   "graph_us": g(lib.pack_ffd), "bytes": 8 * 256 + 4 * 513,
                                   "bound": "latency (sequential first fit)"}
    # doc_ids -> seq_lens bridge: the stress map [64, 32768]
    d4 = dev_t(synth.doc_map_stress(seed))
    Bm, Sm = d4.shape
    np_ = 8192
    r_ = torch.empty(Bm * np_, dtype=torch.int64, device=dev)
    p_ = torch.empty_like(r_)
    pos = torch.empty(Bm * Sm, dtype=torch.int64, device=dev)
    binfo = torch.empty(4, dtype=torch.int32, device=dev)
    bws = torch.zeros(lib.pseq_doc_ids_to_lengths_workspace_size(Bm, Sm), dtype=torch.uint8, device=dev)
    keep += [r_, p_, pos, binfo, bws]
    us = timed(lib.pseq_doc_ids_to_lengths, (P(d4), 4, Bm, Sm, np_, -1000, P(r_), P(p_), P(pos), P(binfo), P(bws),
                                             bws.numel(), sh))
    nbytes = 4 * Bm * Sm + 8 * Bm * Sm + 2 * 8 * Bm * np_
    out["doc_ids_to_seq_lens"] = {"workload": "doc_ids [64,32768] -> seq_lens [64,8192] x2 + positions [64,32768]",
                                  "us": round(us, 2), "graph_us": g(lib.pseq_doc_ids_to_lengths), "bytes": nbytes,
                                  "gbs": round(nbytes / us / 1e3, 1)}
    return out


def link_ceiling(dev, nbytes: int = 256 << 20) -> dict:
    """Host<->device copy bandwidth of this machine from pinned memory: one
    direction at a time, and both at once on two streams (best of 3)."""
    import torch

    h_in = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    h_out = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d_in = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    d_out = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    out = {}
    for mode in ("h2d", "d2h", "both"):
        times = []
        for _ in range(4):
            torch.cuda.synchronize(dev)
            a, b, j = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
                       torch.cuda.Event())
            a.record(s1)
            s2.wait_event(a)
            if mode in ("h2d", "both"):
                with torch.cuda.stream(s1):
                    d_in.copy_(h_in, non_blocking=True)
            if mode in ("d2h", "both"):
                with torch.cuda.stream(s2):
                    h_out.copy_(d_out, non_blocking=True)
            j.record(s2)
            s1.wait_event(j)
            b.record(s1)
            torch.cuda.synchronize(dev)
            times.append(a.elapsed_time(b))
        t = min(times[1:])
        out[f"{mode}_gbs"] = round(nbytes * (2 if mode == "both" else 1) / (t / 1e3) / 1e9, 1)
    return out


def kernel_source_hash() -> str:
    """Hash of the sources the roofline kernel (thd_fused_bulk_kernel) is
    built from -- its translation unit, the shared device header, the C ABI --
    with comments and blank lines removed, so only code changes count."""
    import re

    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "varlen_attention_metadata_gb300", "csrc")
    for path in (os.path.join(csrc, "thd.cu"), os.path.join(csrc, "common.cuh"),
                 os.path.join(ROOT, "include", "pseq.h")):
        with open(path) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()[:16]


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


TRAFFIC_FILE = os.path.join(ROOT, "profiles", "thd_fused_bulk_traffic.json")


def profiled_traffic():
    """DRAM bytes (read + write) per launch of the embedding conversion from
    the committed ncu figures, or None when the kernel's sources changed since
    that capture."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha") != kernel_source_hash():
        return None
    v = rec.get("dram_bytes_per_launch")
    return int(v) if isinstance(v, (int, float)) else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str | None):
        self.samples = []
        self.proc = None
        self.gpu_id = gpu_id
        self.window = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), line.strip()))

    def mark(self, t0, t1):
        self.window = (t0, t1)

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for ts, line in self.samples:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((ts, parts))
        if self.window:
            inside = [r for r in rows if self.window[0] <= r[0] <= self.window[1] + 0.25]
            if inside:
                rows = inside
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(p[1]) for _, p in rows if num(p[1]) is not None]
        mx = [num(p[2]) for _, p in rows if num(p[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, p in rows for i in range(4) if p[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def run_native(args, dist: Dist):
    import torch

    torch.cuda.set_device(dist.local_rank)
    dev = torch.device("cuda", dist.local_rank)
    dist.init("nccl")
    from varlen_attention_metadata_gb300 import build

    if dist.local_rank == 0:
        build.build()
    dist.barrier()

    host = make_inputs(args.seed + dist.rank)
    stream = torch.cuda.Stream(dev)
    side = torch.cuda.Stream(dev)
    step = NativeStep(host, dev, stream, side_stream=side)
    with torch.cuda.stream(stream):
        step.run()
    step.resolve()
    lib = step.lib
    tokens = sum(step.tokens.values())
    per_step_launches = None

    flush_w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    flush_r = torch.zeros(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=dev)

    def flush_l2():
        # write a buffer larger than L2, then read another one so that the
        # dirty lines of the write are evicted here and not inside the next step
        flush_w.zero_()
        flush_r.sum()

    K = args.steps
    W = max(args.warmup, 3)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    gev = [torch.cuda.Event(enable_timing=True) if i % EMB_SAMPLE == 0 else None for i in range(K)]
    with torch.cuda.stream(stream):
        for _ in range(W):
            flush_l2()
            step.run(two_streams=True)
            flush_l2()
            step.run()
    torch.cuda.synchronize(dev)

    # the same step with every call on one stream, for comparison (untimed by the contract)
    K1 = min(K, 500)
    ev1 = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K1)]
    with torch.cuda.stream(stream):
        for i in range(K1):
            flush_l2()
            ev1[i][0].record(stream)
            step.run()
            ev1[i][1].record(stream)
    torch.cuda.synchronize(dev)
    one_stream_ms = statistics.mean(a.elapsed_time(b) for a, b in ev1)
    graph_ms = step_graph_ms(step, dev, stream, flush_l2, K1)

    gpu_id = None
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = None
    clocks = ClockSampler(gpu_id)
    clocks.start()
    time.sleep(0.5)

    dist.barrier()
    torch.cuda.synchronize(dev)
    launches0 = lib.pseq_launch_count()
    t_wall0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(K):
            flush_l2()
            ev[i][0].record(stream)
            step.run(gev[i], two_streams=True)
            ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    dist.barrier()
    launches = lib.pseq_launch_count() - launches0
    per_step_launches = launches // K
    clocks.mark(t_wall0, t_wall1)
    time.sleep(0.3)
    clocks.stop()

    step_ms = [a.elapsed_time(b) for a, b in ev]
    emb_ms = [ev[i][0].elapsed_time(g) for i, g in enumerate(gev) if g is not None]
    total_ms = dist.max(sum(step_ms), dev)
    ms_per_step = total_ms / K
    all_tokens = dist.sum(float(tokens), dev)
    value = all_tokens / (ms_per_step / 1e3)

    # ---- end to end: pinned host inputs in, all outputs back out, every step
    Ke = max(3, min(K, 400))  # about 0.75 s of end-to-end steps: host-side jitter averages out
    # serial: copy in, run, copy out on one stream
    e2e_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    with torch.cuda.stream(stream):
        for _ in range(3):
            step.copy_in()
            step.run()
            step.copy_out()
    torch.cuda.synchronize(dev)
    dist.barrier()
    with torch.cuda.stream(stream):
        e2e_ev[0].record(stream)
        for _ in range(Ke):
            step.copy_in()
            step.run()
            step.copy_out()
        e2e_ev[1].record(stream)
    torch.cuda.synchronize(dev)
    serial_ms = dist.max(e2e_ev[0].elapsed_time(e2e_ev[1]), dev) / Ke
    # pipelined: two buffer sets; copy-in, compute and copy-out on their own streams
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    sets = [step, NativeStep(host, dev, stream, host_pinned=step.pinned)]
    sets[1].run()
    sets[1].resolve()
    in_ready = [torch.cuda.Event() for _ in range(2)]
    out_ready = [torch.cuda.Event() for _ in range(2)]
    freed = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n_steps, start=None, end=None):
        for i in range(n_steps):
            s = sets[i % 2]
            if i >= 2:
                s_in.wait_event(freed[i % 2])
            with torch.cuda.stream(s_in):
                if i == 0 and start is not None:
                    start.record(s_in)
                s.copy_in()
                in_ready[i % 2].record(s_in)
            stream.wait_event(in_ready[i % 2])
            s.run()
            out_ready[i % 2].record(stream)
            s_out.wait_event(out_ready[i % 2])
            with torch.cuda.stream(s_out):
                s.copy_out()
                freed[i % 2].record(s_out)
                if i == n_steps - 1 and end is not None:
                    end.record(s_out)

    pipelined(4)
    torch.cuda.synchronize(dev)
    dist.barrier()
    p_ev = (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    pipelined(Ke, p_ev[0], p_ev[1])
    torch.cuda.synchronize(dev)
    pipe_ms = dist.max(p_ev[0].elapsed_time(p_ev[1]), dev) / Ke

    link = link_ceiling(dev)
    next_rows = time_next_rows(dev, stream, args.seed + dist.rank, flush_l2) if dist.rank == 0 else None

    peak, peak_kind = measured_peak()
    per_config = torch_gpu = launch_floor = None
    if dist.rank == 0:
        host["squeeze_scaled"] = synth.squeeze(args.seed, N=16384)
        host["thd_emb_ragged"] = synth.thd_embeddings_ragged(args.seed)
        per_config = time_per_config(step, host, dev, stream, flush_l2, peak)
        launch_floor = time_launch_floor(dev, stream, flush_l2)
        torch_gpu = time_torch_restatement(host, dev, stream, flush_l2, per_config)
    emb_avg_ms = statistics.mean(emb_ms)
    achieved = step.emb_bytes / (emb_avg_ms / 1e3) / 1e9
    traffic = profiled_traffic()
    cpu = None
    if dist.rank == 0 and dist.world == 1:
        cpu = cpu_baseline(host, budget_s=10.0)
        cpu.update(cpu_description())
        cpu["per_config_full_size"] = oracle_per_config(host)
    dist.barrier()
    if dist.rank == 0:
        line = {
            "metric": METRIC,
            "value": round(value, 1),
            "unit": UNIT,
            "n_gpus": dist.world,
            "steps": K,
            "warmup": W,
            "ms_per_step": round(ms_per_step, 6),
            "higher_is_better": True,
            "scaling": "weak",
            "vs_baseline": None,
            "dtype": "int64",
            "data": "synthetic (seeded generators; shapes and length mixes of packed SFT batches)",
            "config": step_config(step.tokens, step.alg_bytes, dist.world),
            "step_variants": {
                "launch": "direct C ABI calls from prebuilt ctypes arguments; the embedding conversion first "
                          "on the step's stream, the other five calls on a second stream forked from and joined "
                          "back into it",
                "ms_per_step_one_stream": round(one_stream_ms, 6),
                "ms_per_step_graph": round(graph_ms, 6) if graph_ms else None,
                "graph": "the same two-stream step captured once in a CUDA graph and replayed (fork and join "
                         "become graph edges); not the headline, which issues the calls directly",
            },
            "roofline": {
                "kernel": "thd_fused_bulk_kernel via thd_from_batch (bf16 hidden [4,8192,4096] -> [T,4096], cu arrays, mask)",
                "bound": "hbm",
                "achieved": round(achieved, 1),
                "peak": peak,
                "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback",
                "unit": "GB/s",
                "frac": round(achieved / peak, 4),
                "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                "traffic": traffic,
                "algorithmic_bytes_per_launch": step.emb_bytes,
                "avg_launch_us": round(emb_avg_ms * 1e3, 3),
                "launch_us_min_median_max": [round(min(emb_ms) * 1e3, 3), round(statistics.median(emb_ms) * 1e3, 3),
                                             round(max(emb_ms) * 1e3, 3)],
                "timed_as": f"CUDA events on the step's stream: the step's start event (the call is the step's "
                            f"first) to an event recorded right after the call, on every {EMB_SAMPLE}nd timed step "
                            f"({len(emb_ms)} launches)",
                "whole_step": {"achieved": round(sum(step.alg_bytes.values()) / (ms_per_step / 1e3) / 1e9, 1),
                               "frac": round(sum(step.alg_bytes.values()) / (ms_per_step / 1e3) / 1e9 / peak, 4),
                               "what": "algorithmic bytes of all six calls per step over ms_per_step: the step "
                                       "as one bandwidth-bound unit (the dominant kernel shares HBM with the "
                                       "other five calls inside it)"},
            },
            "cpu_baseline": cpu,
            "e2e": {"value": round(all_tokens / (pipe_ms / 1e3), 1), "unit": UNIT,
                    "h2d_bytes_per_step": step.h2d_bytes, "d2h_bytes_per_step": step.d2h_bytes, "steps": Ke,
                    "ms_per_step": round(pipe_ms, 4),
                    "how": "every step copies all inputs in from pinned host memory and all outputs back; "
                           "steps pipelined over two buffer sets (copy-in, compute, copy-out streams)",
                    "serial": {"value": round(all_tokens / (serial_ms / 1e3), 1), "ms_per_step": round(serial_ms, 4),
                               "how": "copy-in, compute, copy-out back to back on one stream"},
                    "link": dict(link, frac_of_both=round((step.h2d_bytes + step.d2h_bytes) / (pipe_ms / 1e3) / 1e9
                                                          / link["both_gbs"], 4),
                                 how="pinned 256 MiB copies through torch (copy engines), best of 3; the pipelined "
                                     "step's host bytes per second over the both-directions figure")},
            "next_rows": next_rows,
            "per_config": per_config,
            "launch_floor": launch_floor,
            "torch_gpu_restatement": {
                "what": "each call restated as plain PyTorch ops on the same GPU (boolean filtering, cumsum, "
                        "nonzero, index gathers; bench-only, not the product path), cold: L2 flushed first, "
                        "host synchronisations inside the timed span",
                "per_config": torch_gpu},
            "gpu_launches": int(launches),
            "gpu_launches_per_step": per_step_launches,
            "clocks": clocks.summary(),
            "wall_s_timed_region": round(t_wall1 - t_wall0, 3),
        }
        print(json.dumps(line), flush=True)
    dist.close()


NOMINAL_HBM_GBS = 8000.0  # the nominal GB300 HBM3e figure (~8 TB/s)

PER_CONFIG = (
    ("map_small", "C0 doc_ids int32 [4,2048] -> cu_seqlens, max_seqlen"),
    ("thd_small", "C0 THD of int64 input_ids/labels/position_ids [4,2048]"),
    ("thd_ids", "C1 THD B=8 S=8192, 64 packs: int64 input_ids, labels, mRoPE [3,8,8192]"),
    ("thd_emb", "C2 THD of bf16 hidden [4,8192,4096]"),
    ("squeeze", "C3 squeeze int64 [256,4096] -> FFD bins x 32768, stretched"),
    ("map_stress", "C4 doc_ids int32 [64,32768], ~250k segments"),
    ("squeeze_scaled", "scaled squeeze (labelled extra, not a config): int64 [16384,4096] -> FFD bins x 32768"),
    ("thd_emb_ragged", "C2 with rows ending short (labelled extra, not a config): bf16 hidden [4,8192,4096], each "
                       "row's last sequence dropped, so T < B*S and every later row moves to a lower stream offset"),
)
ROTATE_MAX_SETS = 4096


def capture_step(step, stream):
    """The two-stream step captured in a CUDA graph (the side stream joins
    the capture through the step's fork event)."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        step.run(two_streams=True)
    return g


def step_graph_ms(step, dev, stream, flush_l2, reps) -> float | None:
    """Mean device time of one replay of the captured step, L2 flushed
    between replays outside the events."""
    import torch

    try:
        g = capture_step(step, stream)
    except RuntimeError:
        return None
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    with torch.cuda.stream(stream):
        for _ in range(3):
            flush_l2()
            g.replay()
        for i in range(reps):
            flush_l2()
            ev[i][0].record(stream)
            g.replay()
            ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    del g
    return ms


def _graph_us(calls, dev, stream, flush_l2, replays=10):
    """Mean device time of one replay of a CUDA graph holding ``calls`` in
    order (L2 flushed before every replay)."""
    import torch

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for fn, args in calls:
            st = fn(*args)
            if st != 0:
                raise RuntimeError(f"status {st} during graph capture")
    ev = []
    with torch.cuda.stream(stream):
        for i in range(3 + replays):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            g.replay()
            b.record(stream)
            if i >= 3:
                ev.append((a, b))
    torch.cuda.synchronize(dev)
    us = statistics.median(a.elapsed_time(b) * 1e3 for a, b in ev)
    del g
    return us


def time_per_config(step, host, dev, stream, flush_l2, peak, warm=20, reps=200) -> dict:
    """Per ABI call of every configuration, three ways:

    - ``cold_us``: median of ``reps`` event-timed calls after ``warm`` warm-up
      calls, L2 flushed before every call (the state a training step sees);
    - ``graph_us``: back-to-back calls on one buffer set, captured in one CUDA
      graph (launch gaps removed; small inputs then sit in L2);
    - ``rotated``: one graph of calls over k independent buffer sets holding
      together at least 4x L2 of algorithmic bytes (k capped at 4096), so that
      HBM, not L2, serves them.
    """
    import torch

    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    out = {}
    for name, label in PER_CONFIG:
        if name not in host:
            continue
        if name in step.alg_bytes:
            base = step
        else:
            base = NativeStep(host, dev, stream, host_pinned=step.pinned, only=(name,))
            with torch.cuda.stream(stream):
                base.run()
            base.resolve()
        fn, args = next((f, a) for n, f, a in base.calls if n == name)
        nbytes = base.alg_bytes[name]
        tokens = base.tokens[name]
        ts = []
        with torch.cuda.stream(stream):
            for i in range(warm + reps):
                flush_l2()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                st = fn(*args)
                b.record(stream)
                if st != 0:
                    raise RuntimeError(f"{name}: status {st}")
                if i >= warm:
                    ts.append((a, b))
        torch.cuda.synchronize(dev)
        cold = statistics.median(a.elapsed_time(b) * 1e3 for a, b in ts)
        G = 200 if nbytes < (64 << 20) else 20
        graph = _graph_us([(fn, args)] * G, dev, stream, flush_l2) / G
        k = int(min(ROTATE_MAX_SETS, max(1, -(-4 * l2 // nbytes))))
        sets = [base] + [NativeStep(host, dev, stream, host_pinned=step.pinned, only=(name,)) for _ in range(k - 1)]
        calls = [next((f, a) for n, f, a in s.calls if n == name) for s in sets]
        rot = _graph_us(calls, dev, stream, flush_l2, replays=5) / k
        del sets, calls
        torch.cuda.empty_cache()
        gbs = nbytes / rot / 1e3
        out[name] = {
            "what": label,
            "algorithmic_bytes": int(nbytes),
            "tokens": int(tokens),
            "cold_us": round(cold, 2),
            "cold_gbs": round(nbytes / cold / 1e3, 1),
            "cold_tokens_per_s": round(tokens / cold * 1e6, 1),
            "graph_us": round(graph, 2),
            "rotated": {"sets": k, "set_bytes_over_l2": round(k * nbytes / l2, 2), "us_per_call": round(rot, 2),
                        "gbs": round(gbs, 1), "frac_of_measured": round(gbs / peak, 4),
                        "frac_of_nominal": round(gbs / NOMINAL_HBM_GBS, 4)},
        }
        if base is not step:
            del base
            torch.cuda.empty_cache()
    return out


def time_launch_floor(dev, stream, flush_l2, warm=20, reps=200) -> dict:
    """The library's smallest launch, timed like the configurations'
    ``cold_us`` and ``graph_us``: ``pseq_from_doc_ids`` on an empty map
    (B = 0), one single-thread kernel writing ``cu_seqlens[0]`` and the info
    block.  What is left of a small call's cold time above this is its own."""
    import torch

    import varlen_attention_metadata_gb300 as v

    lib = v.load_library()
    cu = torch.zeros(16, dtype=torch.int32, device=dev)
    info = torch.zeros(8, dtype=torch.int32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    d = torch.zeros(1, dtype=torch.int32, device=dev)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    args = (P(d), 4, 0, 1, P(cu), P(info), P(ws), ws.numel(), ctypes.c_void_p(stream.cuda_stream))
    fn = lib.pseq_from_doc_ids
    ts = []
    with torch.cuda.stream(stream):
        for i in range(warm + reps):
            flush_l2()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            st = fn(*args)
            b.record(stream)
            if st != 0:
                raise RuntimeError(f"empty map: status {st}")
            if i >= warm:
                ts.append((a, b))
    torch.cuda.synchronize(dev)
    cold = statistics.median(a.elapsed_time(b) * 1e3 for a, b in ts)
    graph = _graph_us([(fn, args)] * 200, dev, stream, flush_l2) / 200
    return {"what": "pseq_from_doc_ids on an empty map: one single-thread kernel, the library's smallest launch, "
                    "timed as the configurations' cold_us and graph_us",
            "cold_us": round(cold, 2), "graph_us": round(graph, 2)}


# ----------------------------------------------------------------------------
# A comparison line: each call restated as plain PyTorch ops on the same GPU
# (boolean filtering, cumsum, nonzero, index gathers), written from what the
# calls compute.  Bench-only and labelled as such; never the product path.
# ----------------------------------------------------------------------------
def torch_doc_ids(d):
    """cu_seqlens (int32) and max_seqlen of a [B, S] document map."""
    import torch

    B, S = d.shape
    starts = torch.ones_like(d, dtype=torch.bool)
    starts[:, 1:] = d[:, 1:] != d[:, :-1]
    idx = starts.reshape(-1).nonzero().squeeze(1)
    cu = torch.cat([idx, idx.new_tensor([B * S])]).to(torch.int32)
    return cu, int((cu[1:] - cu[:-1]).max()) if B * S else 0


def torch_thd(real, padded, S, fields, pad_value=-1000):
    """BSHD -> THD: cu arrays, gathered fields ([planes, B, S, row] tensors
    given as (tensor, planes)), padding mask (True = padding), max_seqlen."""
    import torch

    dev = real.device
    keep = real != pad_value
    r, p = real[keep], padded[keep]
    n = r.numel()
    pz = torch.where(keep, padded, torch.zeros_like(padded))
    off = (pz.cumsum(1) - pz)[keep]
    rows = keep.nonzero()[:, 0]
    cu = torch.zeros(n + 1, dtype=torch.int64, device=dev)
    cup = torch.zeros(n + 1, dtype=torch.int64, device=dev)
    cu[1:] = r.cumsum(0)
    cup[1:] = p.cumsum(0)
    T = int(cup[-1])
    seq = torch.repeat_interleave(torch.arange(n, device=dev), p, output_size=T)
    within = torch.arange(T, device=dev) - cup[:-1][seq]
    src = rows[seq] * S + off[seq] + within
    outs = []
    for x, planes in fields:
        flat = x.reshape(planes, -1, *x.shape[3 if planes > 1 else 2:])
        outs.append(flat[:, src])
    mask = within >= r[seq]
    if n >= 1 and bool((r[:-1] == p[:-1]).all()):
        cu[-1] = T
    max_seqlen = int((cu[1:] - cu[:-1]).max()) if n else 0
    return cu.to(torch.int32), cup.to(torch.int32), outs, mask, max_seqlen


def torch_squeeze(src, real, offsets, members, multiple, capacity, stretch, width, pad_value):
    """The trainer-side squeeze: packed [bins, width], mask (True = padding),
    flat per-bin cu arrays (bin b at offsets[b] + b)."""
    import torch

    dev = src.device
    nb = offsets.numel() - 1
    M = members.numel()
    mem = members.long()
    counts = (offsets[1:] - offsets[:-1]).long()
    bin_of = torch.repeat_interleave(torch.arange(nb, device=dev), counts, output_size=M)
    r = real[mem]
    p = (r + multiple - 1) // multiple * multiple
    ex_p = p.cumsum(0) - p
    ex_r = r.cumsum(0) - r
    first = offsets[:-1].long()
    dst = ex_p - ex_p[first][bin_of]
    totals = torch.zeros(nb, dtype=torch.int64, device=dev).index_add_(0, bin_of, p)
    if bool((totals > capacity).any()) or bool((totals > width).any()):
        raise ValueError("a bin exceeds capacity")
    R = int(r.sum())
    mi = torch.repeat_interleave(torch.arange(M, device=dev), r, output_size=R)
    within = torch.arange(R, device=dev) - ex_r[mi]
    slot = bin_of[mi] * width + dst[mi] + within
    out = torch.full((nb * width,), pad_value, dtype=src.dtype, device=dev)
    out[slot] = src[mem[mi], within]
    mask = torch.ones(nb * width, dtype=torch.bool, device=dev)
    mask[slot] = False
    pos = torch.arange(M, device=dev) + bin_of + 1
    cu = torch.zeros(M + nb, dtype=torch.int64, device=dev)
    cup = torch.zeros(M + nb, dtype=torch.int64, device=dev)
    cu[pos] = r.cumsum(0) - ex_r[first][bin_of]
    cup[pos] = p.cumsum(0) - ex_p[first][bin_of]
    if stretch:
        cup[offsets[1:].long() + torch.arange(nb, device=dev)] = capacity
    return out.view(nb, width), mask.view(nb, width), cu.to(torch.int32), cup.to(torch.int32)


def torch_calls(host: dict, dev) -> dict:
    """One closure per configuration, inputs already on the device."""
    import torch

    def d(a):
        return (a if isinstance(a, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(a))).to(dev)

    calls = {}
    for name in ("map_small", "map_stress"):
        m = d(host[name])
        calls[name] = (lambda m=m: torch_doc_ids(m))
    for name, planes in (("thd_small", 1), ("thd_ids", 3)):
        bt = host[name]
        S = bt["input_ids"].shape[1]
        fields = [(d(bt["input_ids"]), 1), (d(bt["labels"]), 1), (d(bt["position_ids"]), planes)]
        real, pad = d(bt["seq_lens"]), d(bt["seq_lens_padded"])
        calls[name] = (lambda real=real, pad=pad, S=S, fields=fields: torch_thd(real, pad, S, fields))
    emb = host["thd_emb"]
    hid = d(emb["hidden"])
    er, ep = d(emb["seq_lens"]), d(emb["seq_lens_padded"])
    calls["thd_emb"] = lambda: torch_thd(er, ep, hid.shape[1], [(hid, 1)])
    for name in ("squeeze", "squeeze_scaled"):
        if name not in host:
            continue
        c = host[name]
        args = (d(c["src"]), d(c["real_lens"]), d(c["bin_offsets"]), d(c["bin_members"]), c["multiple"],
                c["capacity"], c["stretch"], c["width"], c["pad_value"])
        calls[name] = (lambda args=args: torch_squeeze(*args))
    return calls


def time_torch_restatement(host, dev, stream, flush_l2, per_config, warm=5, reps=30) -> dict:
    """Cold per-call time of the torch restatement (L2 flushed first; the
    host synchronisations its ops need are inside the timed span), beside
    this library's cold time from per_config."""
    import torch

    out = {}
    with torch.cuda.stream(stream):
        calls = torch_calls(host, dev)
        for name, fn in calls.items():
            ts = []
            for i in range(warm + reps):
                flush_l2()
                a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                a.record(stream)
                fn()
                b.record(stream)
                torch.cuda.synchronize(dev)
                if i >= warm:
                    ts.append(a.elapsed_time(b) * 1e3)
            us = statistics.median(ts)
            mine = per_config.get(name, {}).get("cold_us") if per_config else None
            out[name] = {"us": round(us, 2), "pseq_cold_us": mine,
                         "speedup": round(us / mine, 1) if mine else None}
    del calls
    torch.cuda.empty_cache()
    return out


def cpu_description() -> dict:
    model = None
    try:
        res = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10)
        for line in res.stdout.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None:
        model = platform.processor() or platform.machine()
    return {"cpu_model": model, "os_cpu_count": os.cpu_count(), "cores_used": 1}


class OracleStep:
    """One whole step on the host: the oracle's function for every call of the
    step, each on its full-size input.  ``run`` returns, per part, the
    produced (count, stream tokens) -- the same figures the native arm reads
    from each call's info block."""

    def __init__(self, host: dict):
        import oracle
        import torch

        self.host = host

        def map_call(d):
            def run():
                cu, _ = oracle.from_doc_ids(d)
                return len(cu) - 1, d.size
            return run

        def thd_call(bt):
            def run():
                r = oracle.process_input_for_thd(bt)
                return len(r["cu_seqlens"]) - 1, r["total_tokens"]
            return run

        def emb_call(emb):
            h = emb["hidden"].view(torch.int16).numpy()

            def run():
                meta = oracle.thd_meta(emb["seq_lens"], emb["seq_lens_padded"], h.shape[1])
                oracle.thd_gather(h, meta, h.shape[0], h.shape[1])
                oracle.thd_padding_mask(meta["total_tokens"], meta["seq_real"], meta["seq_padded"])
                return meta["num_sequences"], meta["total_tokens"]
            return run

        def squeeze_call(sq):
            def run():
                oracle.pack_squeeze(sq["src"], sq["real_lens"], sq["bin_offsets"], sq["bin_members"], sq["multiple"],
                                    sq["capacity"], sq["stretch"], sq["width"], sq["pad_value"])
                return int(sq["bin_offsets"][-1]), (len(sq["bin_offsets"]) - 1) * sq["width"]
            return run

        self.calls = {"map_small": map_call(host["map_small"]), "thd_small": thd_call(host["thd_small"]),
                      "thd_ids": thd_call(host["thd_ids"]), "thd_emb": emb_call(host["thd_emb"]),
                      "squeeze": squeeze_call(host["squeeze"]), "map_stress": map_call(host["map_stress"])}
        self.extras = {}
        if "squeeze_scaled" in host:
            self.extras["squeeze_scaled"] = squeeze_call(host["squeeze_scaled"])
        if "thd_emb_ragged" in host:
            self.extras["thd_emb_ragged"] = emb_call(host["thd_emb_ragged"])

    def run(self) -> dict:
        return {name: fn() for name, fn in self.calls.items()}

    def tokens_and_bytes(self, produced: dict):
        """Per-part stream tokens and algorithmic bytes of one step."""
        tokens = {k: t for k, (_, t) in produced.items()}
        alg = {k: part_bytes(k, self.host[k], c, t) for k, (c, t) in produced.items()}
        return tokens, alg


def oracle_per_config(host: dict) -> dict:
    """Wall-clock time of the oracle on every configuration at full size,
    single-threaded: median of 5 runs (3 for the embedding batches and the
    scaled squeeze)."""
    step = OracleStep(host)
    out = {}
    for name, fn in list(step.calls.items()) + list(step.extras.items()):
        n = 3 if name in ("thd_emb", "thd_emb_ragged", "squeeze_scaled") else 5
        ts = []
        for _ in range(n):
            t0 = time.perf_counter()
            fn()
            ts.append(time.perf_counter() - t0)
        out[name] = {"ms": round(statistics.median(ts) * 1e3, 3), "runs": n}
    return out


# ----------------------------------------------------------------------------
# oracle arms: cpu_baseline (inside the native run) and --impl reference
# ----------------------------------------------------------------------------
class OracleUnits:
    """The step cut into small independent units for a bounded sample: one
    row of a doc_ids map (rows are independent: every row start is a
    boundary), one row of a THD batch, one sequence of the embedding batch,
    one bin of the squeeze.  ``step(fraction)`` runs that fraction of every
    part's units (at least one each), cycling through them, and returns the
    tokens produced and the seconds spent."""

    def __init__(self, host: dict):
        import oracle
        import torch

        self.oracle = oracle
        self.parts = {}
        for name in ("map_small", "map_stress"):
            m = host[name]
            self.parts[name] = [m[b:b + 1] for b in range(m.shape[0])]
        for name in ("thd_small", "thd_ids"):
            bt = host[name]
            units = []
            for b in range(bt["input_ids"].shape[0]):
                sub = {"input_ids": bt["input_ids"][b:b + 1], "labels": bt["labels"][b:b + 1],
                       "seq_lens": bt["seq_lens"][b:b + 1], "seq_lens_padded": bt["seq_lens_padded"][b:b + 1]}
                pos = bt["position_ids"]
                sub["position_ids"] = pos[:, b:b + 1] if pos.ndim == 3 else pos[b:b + 1]
                units.append(sub)
            self.parts[name] = units
        emb = host["thd_emb"]
        h = emb["hidden"].view(torch.int16).numpy()
        meta = oracle.thd_meta(emb["seq_lens"], emb["seq_lens_padded"], h.shape[1])
        units = []
        for i in range(meta["num_sequences"]):
            b, o, r, p = (int(meta[k][i]) for k in ("seq_row", "seq_off", "seq_real", "seq_padded"))
            units.append({"hidden": h[b:b + 1, o:o + p], "seq_lens": np.array([[r]], np.int64),
                          "seq_lens_padded": np.array([[p]], np.int64)})
        self.parts["thd_emb"] = units
        sq = host["squeeze"]
        self.parts["squeeze"] = [(sq["src"], sq["real_lens"]) + tuple(oracle.bins_to_csr([m])) for m in sq["bins"]]
        self.sq = sq
        self.next = {k: 0 for k in self.parts}

    def _run(self, name, u):
        o = self.oracle
        if name.startswith("map"):
            o.from_doc_ids(u)
            return u.size
        if name == "thd_emb":
            meta = o.thd_meta(u["seq_lens"], u["seq_lens_padded"], u["hidden"].shape[1])
            o.thd_gather(u["hidden"], meta, 1, u["hidden"].shape[1])
            o.thd_padding_mask(meta["total_tokens"], meta["seq_real"], meta["seq_padded"])
            return meta["total_tokens"]
        if name.startswith("thd"):
            return o.process_input_for_thd(u)["total_tokens"]
        src, real, offs, mem = u
        sq = self.sq
        o.pack_squeeze(src, real, offs, mem, sq["multiple"], sq["capacity"], sq["stretch"], sq["width"],
                       sq["pad_value"])
        return sq["width"]

    def step(self, fraction: float):
        tokens, spent = 0, 0.0
        for name, units in self.parts.items():
            for _ in range(max(1, int(round(fraction * len(units))))):
                u = units[self.next[name] % len(units)]
                self.next[name] += 1
                t0 = time.perf_counter()
                tokens += self._run(name, u)
                spent += time.perf_counter() - t0
        return tokens, spent


def cpu_baseline(host: dict, budget_s: float = 10.0) -> dict:
    """The oracle, single-threaded, on whole steps of the same workload for
    about ``budget_s`` seconds (at least two steps)."""
    step = OracleStep(host)
    step.run()  # warm-up
    t0 = time.perf_counter()
    n, tokens = 0, 0
    while time.perf_counter() - t0 < budget_s or n < 2:
        produced = step.run()
        tokens += sum(t for _, t in produced.values())
        n += 1
    wall = time.perf_counter() - t0
    return {"value": round(tokens / wall, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} whole steps (all six calls of the step at full size, one after another) in {wall:.1f} s "
                      f"on one core, after one warm-up step",
            "oracle_ms_per_step": round(wall / n * 1e3, 3)}


REF_BUDGET_S = 150.0  # the reference arm's timed steps stay within about this many seconds


def run_reference(args, dist: Dist):
    """The oracle arm: the oracle as it stands, on one host core, on whole
    steps of the native arm's workload (each step a bounded sample of it when
    --steps is too large to finish within a few minutes).  Under torchrun
    rank 0 alone runs and prints; the other ranks exit without work."""
    if dist.world > 1:
        dist.init("gloo")
        if dist.rank != 0:
            dist.close()
            return
    host = make_inputs(args.seed)
    step = OracleStep(host)
    K, W = args.steps, max(args.warmup, 3)
    t0 = time.perf_counter()
    produced = step.run()
    est = time.perf_counter() - t0
    tokens_by_part, alg = step.tokens_and_bytes(produced)
    step_tokens = sum(tokens_by_part.values())
    whole = (K + W) * est <= REF_BUDGET_S
    if whole:
        for _ in range(W - 1):
            step.run()
        t0 = time.perf_counter()
        for _ in range(K):
            step.run()
        wall = time.perf_counter() - t0
        value = K * step_tokens / wall
        ms_per_step = wall / K * 1e3
        sample = (f"{K} whole steps (all six calls of the step at full size, one after another) after {W} warm-up "
                  f"steps, {wall:.1f} s on one core")
    else:
        units = OracleUnits(host)
        fraction = min(1.0, REF_BUDGET_S / ((K + W) * est))
        for _ in range(W):
            units.step(fraction)
        tokens, spent = 0, 0.0
        t0 = time.perf_counter()
        for _ in range(K):
            tk, sp = units.step(fraction)
            tokens += tk
            spent += sp
        wall = time.perf_counter() - t0
        value = tokens / wall
        ms_per_step = wall / K * 1e3
        sample = (f"{K} steps, each a bounded sample ({fraction:.3f} of the units of every part: map rows, THD rows, "
                  f"embedding sequences, squeeze bins) of the whole step, {wall:.1f} s on one core")
    if dist.world > 1:
        sample += f"; rank 0 of {dist.world} alone (one host core), the other ranks exit without work"
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": dist.world,
        "steps": K,
        "warmup": W,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "int64",
        "data": "synthetic (seeded generators; shapes and length mixes of packed SFT batches)",
        "config": step_config(tokens_by_part, alg, dist.world),
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    if dist.pg is not None:
        dist.close()


def profile_calls(args):
    """The workload for a per-kernel profiler capture: two rounds of every
    configuration's ABI call, the scaled squeeze and the ragged embedding
    batch, then six of each next-row call.  Nothing is timed."""
    import torch

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from varlen_attention_metadata_gb300 import build

    build.build()
    host = make_inputs(args.seed)
    host["squeeze_scaled"] = synth.squeeze(args.seed, N=16384)
    host["thd_emb_ragged"] = synth.thd_embeddings_ragged(args.seed)
    stream = torch.cuda.Stream(dev)
    step = NativeStep(host, dev, stream)
    scaled = NativeStep(host, dev, stream, host_pinned=step.pinned, only=("squeeze_scaled", "thd_emb_ragged"))
    with torch.cuda.stream(stream):
        for _ in range(2):
            for s in (step, scaled):
                for name, fn, a in s.calls:
                    st = fn(*a)
                    if st != 0:
                        raise RuntimeError(f"{name}: status {st}")
    torch.cuda.synchronize(dev)
    step.resolve()
    scaled.resolve()
    time_next_rows(dev, stream, args.seed, lambda: None, reps=1)
    torch.cuda.synchronize(dev)


def main():
    args = parse_args()
    if args.profile_calls:
        profile_calls(args)
        return
    dist = Dist()
    if args.gpus > 1 and dist.world == 1:
        sys.exit("bench.py --gpus N > 1 must be launched with torchrun (one process per GPU)")
    if args.impl == "reference":
        run_reference(args, dist)
    else:
        run_native(args, dist)


if __name__ == "__main__":
    main()

"""Plain CPU oracle for the packed-sequence metadata path.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
product package never imports it, and it imports nothing from the product
package: the two share no code, header, helper or constant.

The arithmetic lives in ``pseq_oracle.c`` (plain single-threaded loops, int64
throughout).  This module only compiles that file with the host C compiler,
marshals numpy arrays through ``ctypes`` and turns the oracle's own status
codes into exceptions:

* ``OracleValueError``    malformed lengths or layout
* ``OracleCapacityError`` a bin that does not fit its capacity or row width
* ``ValueError``          an argument the caller could have checked up front

Pages followed (each C function cites its section):

* NeMo AutoModel API reference, ``nemo_automodel.components.datasets.packed_seq``
* NeMo AutoModel v0.5 API reference, ``nemo_automodel.components.distributed.thd_utils``
* "Who packs the sequences: the loader, or the trainer?" (NeMo-RL #4105 explainer)
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pseq_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")

_ORC_OK, _ORC_VALUE, _ORC_CAPACITY = 0, 3, 4

_lock = threading.Lock()
_lib = None


class OracleValueError(ValueError):
    """The oracle found malformed lengths or a malformed layout."""


class OracleCapacityError(ValueError):
    """A bin's padded total exceeds its capacity or the output row width."""


def compile_library(source: str = SOURCE, out_dir: str = BUILD_DIR, strict: bool = True) -> str:
    """Compile ``source`` into a shared library and return its path.

    The file name carries a hash of the source text, the flags and the
    machine, so a stale or foreign-architecture build is never reused.
    ``strict`` turns warnings into errors (off for deliberately broken copies).
    """
    with open(source, "rb") as f:
        text = f.read()
    flags = ["-O2", "-std=c11", "-shared", "-fPIC", "-Wall"] + (["-Werror"] if strict else [])
    key = hashlib.sha256(text + " ".join(flags).encode() + os.uname().machine.encode()).hexdigest()[:16]
    os.makedirs(out_dir, exist_ok=True)
    path = os.path.join(out_dir, f"liboracle_{key}.so")
    if not os.path.exists(path):
        tmp = f"{path}.{os.getpid()}.tmp"
        subprocess.run(["gcc", *flags, "-o", tmp, source], check=True)
        os.replace(tmp, path)
    return path


def _declare(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    I32 = ctypes.c_int
    lib.oracle_from_doc_ids.restype = I64
    lib.oracle_from_doc_ids.argtypes = [P, I32, I64, I64, P, P]
    lib.oracle_thd_meta.restype = I32
    lib.oracle_thd_meta.argtypes = [P, P, I64, I64, I64, I64, I32, P, P, P, P, P, P, P, P, P, P]
    lib.oracle_thd_gather.restype = None
    lib.oracle_thd_gather.argtypes = [P, P, I32, I64, I64, I64, I64, I64, P, P, P, P, I64]
    lib.oracle_thd_padding_mask.restype = I32
    lib.oracle_thd_padding_mask.argtypes = [I64, P, P, I64, P]
    lib.oracle_mask_from_token_ids.restype = I32
    lib.oracle_mask_from_token_ids.argtypes = [P, I32, I64, I64, P]
    lib.oracle_ffd.restype = I32
    lib.oracle_ffd.argtypes = [P, I64, I64, P, P, P]
    lib.oracle_doc_ids_to_lengths.restype = I32
    lib.oracle_doc_ids_to_lengths.argtypes = [P, I32, I64, I64, I64, I64, P, P, P]
    lib.oracle_pack_squeeze.restype = I32
    lib.oracle_pack_squeeze.argtypes = [P, I64, I64, I32, P, P, P, I64, I64, I64, I32, I64, I64,
                                        P, P, P, P, P]
    return lib


def load_library(path: str | None = None):
    """Load (building first if needed) the oracle library.

    With ``path`` given, load that file instead of the default build; the
    mutation tests use this to load deliberately broken copies.
    """
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(compile_library()))
        return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _check(status: int):
    if status == _ORC_VALUE:
        raise OracleValueError("malformed lengths or layout")
    if status == _ORC_CAPACITY:
        raise OracleCapacityError("bin exceeds capacity or row width")
    if status != _ORC_OK:
        raise RuntimeError(f"oracle returned unknown status {status}")


# --------------------------------------------------------------------------
# O1 packed_seq_params_from_doc_ids
# --------------------------------------------------------------------------
def from_doc_ids(doc_ids: np.ndarray, lib=None):
    """Segment boundaries of a neat-packing document map.

    Returns ``(cu_seqlens int32 [num_segments+1], max_seqlen int)``.
    Follows packed_seq: ``packed_seq_params_from_doc_ids``.
    """
    lib = lib or load_library()
    d = np.ascontiguousarray(doc_ids)
    if d.ndim != 2:
        raise ValueError("doc_ids must be [batch, sequence]")
    if d.dtype not in (np.int32, np.int64):
        raise ValueError("doc_ids must be int32 or int64")
    B, S = d.shape
    cu = np.zeros(B * S + 1, dtype=np.int32)
    mx = np.zeros(1, dtype=np.int32)
    nseg = lib.oracle_from_doc_ids(_ptr(d), d.dtype.itemsize, B, S, _ptr(cu), _ptr(mx))
    return cu[: nseg + 1].copy(), int(mx[0])


# --------------------------------------------------------------------------
# O2 + O3 + O4 process_input_for_thd
# --------------------------------------------------------------------------
def thd_meta(seq_lens: np.ndarray, seq_lens_padded: np.ndarray | None, S: int,
             pad_value: int = -1000, absorb: bool = True, lib=None) -> dict:
    """Filtered lengths, cumulative boundaries, absorption, flags.

    Follows thd_utils: ``process_input_for_thd`` (description, Example,
    Returns).  Returns a dict with ``cu_seqlens``, ``cu_seqlens_padded``
    (int32 ``[n+1]``), ``max_seqlen``, ``pad_between_seqs``, ``total_tokens``
    and the per-sequence source layout ``seq_row``, ``seq_off``,
    ``seq_real``, ``seq_padded``.
    """
    lib = lib or load_library()
    real = np.ascontiguousarray(seq_lens, dtype=np.int64)
    if real.ndim != 2:
        raise ValueError("seq_lens must be [batch, num_packs]")
    padded = None
    if seq_lens_padded is not None:
        padded = np.ascontiguousarray(seq_lens_padded, dtype=np.int64)
        if padded.shape != real.shape:
            raise ValueError("seq_lens_padded must match seq_lens")
    B, P = real.shape
    cap = B * P
    cu = np.zeros(cap + 1, np.int32)
    cup = np.zeros(cap + 1, np.int32)
    row = np.zeros(max(cap, 1), np.int64)
    off = np.zeros(max(cap, 1), np.int64)
    sr = np.zeros(max(cap, 1), np.int64)
    sp = np.zeros(max(cap, 1), np.int64)
    n = np.zeros(1, np.int64)
    T = np.zeros(1, np.int64)
    mx = np.zeros(1, np.int32)
    pbs = np.zeros(1, np.int32)
    st = lib.oracle_thd_meta(_ptr(real), _ptr(padded), B, S, P, pad_value, int(bool(absorb)),
                             _ptr(cu), _ptr(cup), _ptr(row), _ptr(off), _ptr(sr), _ptr(sp),
                             _ptr(n), _ptr(T), _ptr(mx), _ptr(pbs))
    _check(st)
    k = int(n[0])
    return {
        "cu_seqlens": cu[: k + 1].copy(),
        "cu_seqlens_padded": cup[: k + 1].copy(),
        "max_seqlen": int(mx[0]),
        "pad_between_seqs": bool(pbs[0]),
        "total_tokens": int(T[0]),
        "num_sequences": k,
        "seq_row": row[:k].copy(),
        "seq_off": off[:k].copy(),
        "seq_real": sr[:k].copy(),
        "seq_padded": sp[:k].copy(),
    }


def thd_gather(src: np.ndarray, meta: dict, B: int, S: int, planes: int = 1, lib=None) -> np.ndarray:
    """Concatenate every kept sequence of ``src`` into the flat THD stream.

    ``src`` is laid out ``[planes, B, S, *row]`` (``planes`` may be folded
    away when 1).  Returns ``[planes, T, *row]`` (``[T, *row]`` when the input
    had no plane axis).  Follows thd_utils: ``process_input_for_thd``
    (description, Returns).
    """
    lib = lib or load_library()
    a = np.ascontiguousarray(src)
    has_planes = planes != 1
    if planes == 1:
        if a.shape[:2] != (B, S):
            raise ValueError("source must be [B, S, ...] when planes == 1")
        row_shape = a.shape[2:]
    else:
        if a.shape[:3] != (planes, B, S):
            raise ValueError("source must be [planes, B, S, ...]")
        row_shape = a.shape[3:]
    row_elems = int(np.prod(row_shape)) if row_shape else 1
    T = meta["total_tokens"]
    out_shape = ((planes,) if has_planes else ()) + (T,) + tuple(row_shape)
    out = np.zeros(out_shape, dtype=a.dtype)
    n = meta["num_sequences"]
    row = np.ascontiguousarray(meta["seq_row"], np.int64)
    off = np.ascontiguousarray(meta["seq_off"], np.int64)
    pad = np.ascontiguousarray(meta["seq_padded"], np.int64)
    cup = np.ascontiguousarray(meta["cu_seqlens_padded"], np.int32)
    if n > 0 and T > 0:
        lib.oracle_thd_gather(_ptr(a), _ptr(out), a.dtype.itemsize, planes, row_elems, B, S, n,
                              _ptr(row), _ptr(off), _ptr(pad), _ptr(cup), T)
    return out


def thd_padding_mask(total_tokens: int, valid_seq_lens: np.ndarray,
                     valid_seq_lens_padded: np.ndarray | None, lib=None) -> np.ndarray:
    """Layout-derived padding mask, True marks padding.

    Follows thd_utils: ``_thd_padding_mask``.
    """
    lib = lib or load_library()
    real = np.ascontiguousarray(valid_seq_lens, np.int64).reshape(-1)
    padded = None
    if valid_seq_lens_padded is not None:
        padded = np.ascontiguousarray(valid_seq_lens_padded, np.int64).reshape(-1)
        if padded.shape != real.shape:
            raise ValueError("valid_seq_lens_padded must match valid_seq_lens")
    if total_tokens < 0:
        raise ValueError("total_tokens must be >= 0")
    mask = np.zeros(max(total_tokens, 1), np.uint8)
    _check(lib.oracle_thd_padding_mask(total_tokens, _ptr(real), _ptr(padded), real.size, _ptr(mask)))
    return mask[:total_tokens].astype(bool)


def process_input_for_thd(batch: dict, seq_lens_padding_value: int = -1000,
                          absorb: bool = True, lib=None) -> dict:
    """Whole BSHD -> THD conversion of a batch of numpy arrays.

    Follows thd_utils: ``process_input_for_thd``.  ``position_ids`` may be
    ``[B,S]`` or mRoPE ``[n_rope,B,S]`` (returned as ``[n_rope,1,T]``);
    ``input_ids`` may be ``[B,S]`` or embeddings ``[B,S,H]``.
    """
    lib = lib or load_library()
    ids = batch["input_ids"]
    B, S = ids.shape[0], ids.shape[1]
    meta = thd_meta(batch["seq_lens"], batch.get("seq_lens_padded"), S,
                    seq_lens_padding_value, absorb, lib=lib)
    out = {k: v for k, v in batch.items() if not isinstance(v, np.ndarray)}
    out["input_ids"] = thd_gather(ids, meta, B, S, lib=lib)
    if "labels" in batch:
        out["labels"] = thd_gather(batch["labels"], meta, B, S, lib=lib)
    pos = batch.get("position_ids")
    if pos is not None:
        if pos.ndim == 3:
            g = thd_gather(pos, meta, B, S, planes=pos.shape[0], lib=lib)
            out["position_ids"] = g.reshape(pos.shape[0], 1, meta["total_tokens"])
        else:
            out["position_ids"] = thd_gather(pos, meta, B, S, lib=lib)
    out["cu_seqlens"] = meta["cu_seqlens"]
    if batch.get("seq_lens_padded") is not None:
        out["cu_seqlens_padded"] = meta["cu_seqlens_padded"]
    out["pad_between_seqs"] = meta["pad_between_seqs"]
    out["max_seqlen"] = meta["max_seqlen"]
    out["padding_mask"] = thd_padding_mask(meta["total_tokens"], meta["seq_real"],
                                           meta["seq_padded"] if batch.get("seq_lens_padded") is not None else None,
                                           lib=lib)
    out["total_tokens"] = meta["total_tokens"]
    return out


# --------------------------------------------------------------------------
# O5 trainer-side squeeze
# --------------------------------------------------------------------------
def bins_to_csr(bins):
    """Convert a list of lists of row indices into ``(offsets, members)``."""
    offsets = np.zeros(len(bins) + 1, np.int32)
    members = []
    for b, members_b in enumerate(bins):
        members.extend(int(i) for i in members_b)
        offsets[b + 1] = len(members)
    return offsets, np.asarray(members, np.int32)


def pack_squeeze(src: np.ndarray, real_lens: np.ndarray, bin_offsets: np.ndarray,
                 bin_members: np.ndarray, multiple: int, capacity: int,
                 stretch_to_capacity: bool, width: int, pad_value: int = 0, lib=None) -> dict:
    """Concatenate the sources of each bin end to end, padded to ``multiple``.

    Follows "Who packs the sequences": "Trainer packs" and "Loader packs".
    Returns ``packed`` ``[num_bins, width]``, the per-bin ``cu_seqlens`` and
    ``cu_seqlens_padded`` (lists of int32 arrays), ``padding_mask`` and
    ``max_total`` (the widest bin before stretching).
    """
    lib = lib or load_library()
    a = np.ascontiguousarray(src)
    if a.ndim != 2:
        raise ValueError("src must be [N, W]")
    N, W = a.shape
    real = np.ascontiguousarray(real_lens, np.int64).reshape(-1)
    offs = np.ascontiguousarray(bin_offsets, np.int32).reshape(-1)
    mem = np.ascontiguousarray(bin_members, np.int32).reshape(-1)
    if real.size != N:
        raise ValueError("real_lens must have one entry per source row")
    if multiple < 1 or capacity < 0 or width < 0:
        raise ValueError("multiple must be >= 1, capacity and width >= 0")
    if stretch_to_capacity and width < capacity:
        raise ValueError("stretching to capacity needs width >= capacity")
    if offs.size < 1:
        raise ValueError("bin_offsets needs num_bins + 1 entries")
    num_bins = offs.size - 1
    M = int(offs[-1])
    out = np.zeros((num_bins, width), dtype=a.dtype)
    mask = np.zeros((num_bins, width), np.uint8)
    cu = np.zeros(M + num_bins + 1, np.int32)
    cup = np.zeros(M + num_bins + 1, np.int32)
    mt = np.zeros(1, np.int64)
    mem_arg = mem if mem.size else np.zeros(1, np.int32)
    st = lib.oracle_pack_squeeze(_ptr(a), N, W, a.dtype.itemsize, _ptr(real), _ptr(offs), _ptr(mem_arg),
                                 num_bins, multiple, capacity, int(bool(stretch_to_capacity)), width,
                                 pad_value, _ptr(out), _ptr(cu), _ptr(cup), _ptr(mask), _ptr(mt))
    _check(st)
    cus = [cu[offs[b] + b: offs[b + 1] + b + 1].copy() for b in range(num_bins)]
    cups = [cup[offs[b] + b: offs[b + 1] + b + 1].copy() for b in range(num_bins)]
    return {
        "packed": out,
        "cu_seqlens": cus,
        "cu_seqlens_padded": cups,
        "padding_mask": mask.astype(bool),
        "max_total": int(mt[0]),
        "cu_flat": cu[: M + num_bins].copy(),
        "cu_padded_flat": cup[: M + num_bins].copy(),
    }


# --------------------------------------------------------------------------
# O6 thd_padding_mask_from_token_ids
# --------------------------------------------------------------------------
def mask_from_token_ids(input_ids: np.ndarray, padding_token_id: int, lib=None) -> np.ndarray:
    """Value-compare padding mask, rejecting a pad id that is also content.

    Follows thd_utils: ``thd_padding_mask_from_token_ids``.  Raises
    ``OracleValueError`` when a pad token is followed by a non-pad token.
    """
    lib = lib or load_library()
    ids = np.ascontiguousarray(input_ids).reshape(-1)
    if ids.dtype not in (np.int32, np.int64):
        raise ValueError("input_ids must be int32 or int64")
    mask = np.zeros(max(ids.size, 1), np.uint8)
    _check(lib.oracle_mask_from_token_ids(_ptr(ids if ids.size else np.zeros(1, ids.dtype)), ids.dtype.itemsize,
                                          ids.size, padding_token_id, _ptr(mask)))
    return mask[:ids.size].astype(bool)


# --------------------------------------------------------------------------
# O7 first-fit-decreasing bins
# --------------------------------------------------------------------------
def ffd(sizes: np.ndarray, capacity: int, lib=None):
    """First-fit-decreasing bins of ``sizes`` at ``capacity``.

    Follows "Who packs the sequences" (get_packer, First Fit Decreasing).
    Returns ``(bin_offsets int32 [nb+1], bin_members int32 [n])``.
    """
    lib = lib or load_library()
    sz = np.ascontiguousarray(sizes, np.int64).reshape(-1)
    n = sz.size
    offs = np.zeros(n + 2, np.int32)
    mem = np.zeros(max(n, 1), np.int32)
    nb = np.zeros(1, np.int64)
    _check(lib.oracle_ffd(_ptr(sz if n else np.zeros(1, np.int64)), n, capacity, _ptr(offs), _ptr(mem), _ptr(nb)))
    k = int(nb[0])
    return offs[: k + 1].copy(), mem[:n].copy()


# --------------------------------------------------------------------------
# O8 doc_ids -> pack lengths and positions
# --------------------------------------------------------------------------
def doc_ids_to_lengths(doc_ids: np.ndarray, num_packs: int, pad_value: int = -1000, lib=None) -> dict:
    """seq_lens, seq_lens_padded [B, num_packs] and position_ids [B, S] of a
    neat-packing map (see the C function for the readings).  Raises
    ``OracleCapacityError`` when a row holds more than num_packs sequences."""
    lib = lib or load_library()
    d = np.ascontiguousarray(doc_ids)
    if d.ndim != 2 or d.dtype not in (np.int32, np.int64):
        raise ValueError("doc_ids must be int32 or int64 [B, S]")
    B, S = d.shape
    real = np.zeros(max(B * num_packs, 1), np.int64)
    padded = np.zeros(max(B * num_packs, 1), np.int64)
    pos = np.zeros(max(B * S, 1), np.int64)
    _check(lib.oracle_doc_ids_to_lengths(_ptr(d if d.size else np.zeros(1, d.dtype)), d.dtype.itemsize, B, S,
                                         num_packs, pad_value, _ptr(real), _ptr(padded), _ptr(pos)))
    return {"seq_lens": real[: B * num_packs].reshape(B, num_packs),
            "seq_lens_padded": padded[: B * num_packs].reshape(B, num_packs),
            "position_ids": pos[: B * S].reshape(B, S)}


# --------------------------------------------------------------------------
# O9 split_batch_into_thd_chunks
# --------------------------------------------------------------------------
def split_batch_into_thd_chunks(batch: dict, num_chunks: int, seq_lens_padding_value: int = -1000,
                                absorb: bool = True, lib=None) -> dict:
    """thd_utils ``split_batch_into_thd_chunks``: split the batch along its
    first axis into ``num_chunks`` equal chunks, run process_input_for_thd on
    each, stack every tensor result on a new leading axis, and pad the
    cu_seqlens arrays to one length with ``seq_lens_padding_value``.

    Readings: chunks whose streams have different lengths cannot be stacked
    (``OracleValueError``); per-chunk scalars (max_seqlen, pad_between_seqs,
    total_tokens) become arrays of length num_chunks; num_chunks <= 1 returns
    process_input_for_thd unchanged.
    """
    lib = lib or load_library()
    if num_chunks <= 1:
        return process_input_for_thd(batch, seq_lens_padding_value, absorb, lib=lib)
    B = batch["input_ids"].shape[0]
    if B % num_chunks:
        raise ValueError("num_chunks must evenly divide the batch size")
    Bc = B // num_chunks
    parts = []
    for c in range(num_chunks):
        sub = {}
        for k, v in batch.items():
            if not isinstance(v, np.ndarray):
                sub[k] = v
            elif k == "position_ids" and v.ndim == 3:
                sub[k] = v[:, c * Bc:(c + 1) * Bc]
            else:
                sub[k] = v[c * Bc:(c + 1) * Bc]
        parts.append(process_input_for_thd(sub, seq_lens_padding_value, absorb, lib=lib))
    if len({p["total_tokens"] for p in parts}) != 1:
        raise OracleValueError("chunks produce streams of different lengths and cannot be stacked")
    out = {k: v for k, v in parts[0].items() if not isinstance(v, (np.ndarray, bool, int, np.bool_))}
    for k in ("input_ids", "labels", "position_ids", "padding_mask"):
        if k in parts[0]:
            out[k] = np.stack([p[k] for p in parts])
    for k in ("cu_seqlens", "cu_seqlens_padded"):
        if k in parts[0]:
            width = max(p[k].size for p in parts)
            rows = np.full((num_chunks, width), seq_lens_padding_value, np.int32)
            for c, p in enumerate(parts):
                rows[c, : p[k].size] = p[k]
            out[k] = rows
    out["max_seqlen"] = np.array([p["max_seqlen"] for p in parts], np.int32)
    out["pad_between_seqs"] = np.array([p["pad_between_seqs"] for p in parts], bool)
    out["total_tokens"] = parts[0]["total_tokens"]
    out["num_sequences"] = np.array([p["cu_seqlens"].size - 1 for p in parts], np.int32)
    return out

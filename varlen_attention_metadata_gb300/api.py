"""Torch-facing binding of libpseq.

Two layers, both argument marshalling only (every step runs in the CUDA
kernels behind the C ABI):

* the C entry points under their own names -- ``pseq_from_doc_ids``,
  ``thd_from_batch``, ``thd_meta``, ``thd_gather``, ``thd_padding_mask``,
  ``pack_squeeze`` -- taking CUDA tensors, enqueueing on the current stream
  and returning device tensors sized for the worst case plus the 16-byte
  ``info`` block, without synchronising;
* the pages' functions -- ``packed_seq_params_from_doc_ids``,
  ``to_flash_attention_kwargs`` (NeMo AutoModel packed_seq),
  ``process_input_for_thd``, ``_thd_padding_mask`` (NeMo AutoModel v0.5
  thd_utils) and ``squeeze_bins`` (the trainer-side squeeze of "Who packs the
  sequences") -- which read the info block back (one small device-to-host
  copy), raise on device-reported errors and narrow the outputs to their
  exact sizes.

Tensors must be contiguous and on one CUDA device; nothing is converted or
moved implicitly, and there is no CPU path.
"""
from __future__ import annotations

import ctypes
import math
import threading
from dataclasses import dataclass

import torch

from . import _lib

__all__ = [
    "PackedSeqParams",
    "thd_chunks_from_batch",
    "thd_mask_from_token_ids",
    "pack_ffd",
    "pseq_doc_ids_to_lengths",
    "split_batch_into_thd_chunks",
    "thd_padding_mask_from_token_ids",
    "first_fit_decreasing",
    "doc_ids_to_seq_lens",
    "pseq_from_doc_ids",
    "thd_from_batch",
    "thd_meta",
    "thd_gather",
    "thd_padding_mask",
    "pack_squeeze",
    "packed_seq_params_from_doc_ids",
    "to_flash_attention_kwargs",
    "process_input_for_thd",
    "_thd_padding_mask",
    "squeeze_bins",
    "check_info",
]


# ----------------------------------------------------------------------------
# marshalling helpers
# ----------------------------------------------------------------------------
def _p(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device: torch.device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _require_cuda(name: str, t: torch.Tensor, dtypes=None, device=None) -> torch.Tensor:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be on a CUDA device (there is no CPU path), got {t.device}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if dtypes is not None and t.dtype not in dtypes:
        raise TypeError(f"{name} must have dtype in {dtypes}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


class _WorkspaceCache:
    """One workspace buffer per (kind, device, stream), grown on demand.

    Kinds in ``ZEROED`` are zero-filled when allocated: those kernels need
    a zeroed workspace at first use and leave it fit for the next call (the
    scan's stamped slots, the others' counters back at zero), so reuse on
    the same stream needs no further clearing.  Each kind has its own buffer, so
    one kernel's scratch never lands in another's.  Other kinds hold
    per-call scratch.
    """

    ZEROED = ("scan", "token_mask", "squeeze", "bridge")

    def __init__(self):
        self._bufs: dict = {}
        self._lock = threading.Lock()

    def get(self, kind: str, nbytes: int, device: torch.device) -> torch.Tensor:
        stream = torch.cuda.current_stream(device).cuda_stream
        key = (kind, device.index, stream)
        with self._lock:
            buf = self._bufs.get(key)
            if buf is None or buf.numel() < nbytes:
                size = max(256, 1 << max(8, math.ceil(math.log2(max(nbytes, 1)))))
                buf = (torch.zeros if kind in self.ZEROED else torch.empty)(size, dtype=torch.uint8, device=device)
                self._bufs[key] = buf
            return buf


_workspaces = _WorkspaceCache()


def _new_info(device) -> torch.Tensor:
    """Device block: pseq_info (16 bytes) followed by one flag byte."""
    return torch.empty(32, dtype=torch.uint8, device=device)


def _info_view(block: torch.Tensor) -> torch.Tensor:
    return block[:16].view(torch.int32)


def check_info(block: torch.Tensor, what: str) -> tuple[int, int, int, int]:
    """Read the info block back (synchronises) and raise on a device error.

    Malformed input and capacity problems raise ``ValueError``, as the pages'
    functions do; a bounded wait that gave up raises ``RuntimeError``.
    Returns ``(status, count, max_seqlen, total)``.
    """
    st, count, mx, total = _info_view(block).tolist()
    if st == _lib.PSEQ_OK:
        return st, count, mx, total
    name = _lib.STATUS_NAMES.get(st, str(st))
    if st in (_lib.PSEQ_ERR_VALUE, _lib.PSEQ_ERR_CAPACITY):
        raise ValueError(f"{what}: device reported {name}")
    raise RuntimeError(f"{what}: device reported {name}")


# ----------------------------------------------------------------------------
# C entry points, same names (asynchronous)
# ----------------------------------------------------------------------------
def pseq_from_doc_ids(doc_ids: torch.Tensor, cu_seqlens: torch.Tensor | None = None,
                      info: torch.Tensor | None = None):
    """Enqueue the segment scan of ``doc_ids`` [B, S] (int32 or int64).

    Returns ``(cu_seqlens, info)``: int32 ``[B*S+1]`` capacity (the first
    ``count + 1`` entries are valid) and the 32-byte info block.
    """
    lib = _lib.load()
    _require_cuda("doc_ids", doc_ids, (torch.int32, torch.int64))
    if doc_ids.dim() != 2:
        raise ValueError("doc_ids must be [batch, sequence]")
    dev = doc_ids.device
    B, S = doc_ids.shape
    if cu_seqlens is None:
        cu_seqlens = torch.empty(B * S + 1, dtype=torch.int32, device=dev)
    if info is None:
        info = _new_info(dev)
    nbytes = lib.pseq_from_doc_ids_workspace_size(B, S)
    ws = _workspaces.get("scan", nbytes, dev)
    _lib.check(lib.pseq_from_doc_ids(_p(doc_ids), doc_ids.element_size(), B, S, _p(cu_seqlens), _p(info),
                                     _p(ws), ws.numel(), _stream(dev)))
    return cu_seqlens, info


def _fields(tensors, B: int, S: int, dev):
    """Build pseq_field entries and worst-case destination buffers.

    Each entry of ``tensors`` is ``(src, planes)`` with src laid out
    [planes, B, S, *row] (planes folded away when 1).
    """
    arr = (_lib.PseqField * max(1, len(tensors)))()
    dsts = []
    for i, (src, planes) in enumerate(tensors):
        _require_cuda("field", src, device=dev)
        lead = (planes, B, S) if planes > 1 else (B, S)
        if tuple(src.shape[:len(lead)]) != lead:
            raise ValueError(f"field {i} has shape {tuple(src.shape)}, expected leading {lead}")
        row = tuple(src.shape[len(lead):])
        row_elems = math.prod(row) if row else 1
        dst = torch.empty(planes * B * S * row_elems, dtype=src.dtype, device=dev)
        arr[i].src = src.data_ptr()
        arr[i].dst = dst.data_ptr()
        arr[i].elem_bytes = src.element_size()
        arr[i].planes = planes
        arr[i].row_elems = row_elems
        dsts.append((dst, planes, row))
    return arr, dsts


def thd_from_batch(seq_lens: torch.Tensor, seq_lens_padded: torch.Tensor | None, S: int,
                   fields=(), pad_value: int = -1000, absorb_trailing_pad: bool = True,
                   want_mask: bool = True):
    """Enqueue the whole BSHD -> THD conversion.

    ``fields`` is a sequence of ``(src, planes)``.  Returns a dict of device
    tensors sized for the worst case: ``cu_seqlens``, ``cu_seqlens_padded``
    (or None), ``padding_mask`` (or None), ``dst`` (list of ``(flat buffer,
    planes, row shape)``) and the info block ``info`` (pad_between_seqs is
    byte 16 of it).
    """
    lib = _lib.load()
    _require_cuda("seq_lens", seq_lens, (torch.int64,))
    dev = seq_lens.device
    if seq_lens.dim() != 2:
        raise ValueError("seq_lens must be [batch, num_packs]")
    if seq_lens_padded is not None:
        _require_cuda("seq_lens_padded", seq_lens_padded, (torch.int64,), dev)
        if seq_lens_padded.shape != seq_lens.shape:
            raise ValueError("seq_lens_padded must have the shape of seq_lens")
    B, P = seq_lens.shape
    if len(fields) > _lib.PSEQ_MAX_FIELDS:
        raise ValueError(f"at most {_lib.PSEQ_MAX_FIELDS} fields")
    arr, dsts = _fields(fields, B, S, dev)
    cu = torch.empty(B * P + 1, dtype=torch.int32, device=dev)
    cup = torch.empty(B * P + 1, dtype=torch.int32, device=dev) if seq_lens_padded is not None else None
    mask = torch.empty(B * S, dtype=torch.bool, device=dev) if want_mask else None
    info = _new_info(dev)
    nbytes = lib.thd_workspace_size(B, P)
    ws = _workspaces.get("thd", nbytes, dev)
    _lib.check(lib.thd_from_batch(_p(seq_lens), _p(seq_lens_padded), B, S, P, pad_value,
                                  1 if absorb_trailing_pad else 0, arr if fields else None, len(fields),
                                  _p(cu), _p(cup), _p(mask), ctypes.c_void_p(info.data_ptr() + 16), _p(info),
                                  _p(ws), ws.numel(), _stream(dev)))
    return {"cu_seqlens": cu, "cu_seqlens_padded": cup, "padding_mask": mask, "dst": dsts, "info": info,
            "workspace": ws}


def thd_meta(seq_lens, seq_lens_padded, S: int, pad_value: int = -1000, absorb_trailing_pad: bool = True):
    """Enqueue only the metadata half of the conversion (see thd_from_batch)."""
    lib = _lib.load()
    _require_cuda("seq_lens", seq_lens, (torch.int64,))
    dev = seq_lens.device
    if seq_lens_padded is not None:
        _require_cuda("seq_lens_padded", seq_lens_padded, (torch.int64,), dev)
    B, P = seq_lens.shape
    cu = torch.empty(B * P + 1, dtype=torch.int32, device=dev)
    cup = torch.empty(B * P + 1, dtype=torch.int32, device=dev) if seq_lens_padded is not None else None
    info = _new_info(dev)
    # the layout stays in this workspace until thd_gather reads it, so it is
    # the caller's (held in the returned dict), not the per-stream cached one
    # that the next conversion on the stream would overwrite
    ws = torch.empty(lib.thd_workspace_size(B, P), dtype=torch.uint8, device=dev)
    _lib.check(lib.thd_meta(_p(seq_lens), _p(seq_lens_padded), B, S, P, pad_value, 1 if absorb_trailing_pad else 0,
                            _p(cu), _p(cup), ctypes.c_void_p(info.data_ptr() + 16), _p(info), _p(ws), ws.numel(),
                            _stream(dev)))
    return {"cu_seqlens": cu, "cu_seqlens_padded": cup, "info": info, "workspace": ws, "B": B, "S": S, "P": P}


def thd_gather(meta: dict, fields=(), want_mask: bool = True):
    """Enqueue the gather half after ``thd_meta`` (same stream)."""
    lib = _lib.load()
    B, S, P, ws = meta["B"], meta["S"], meta["P"], meta["workspace"]
    dev = ws.device
    arr, dsts = _fields(fields, B, S, dev)
    mask = torch.empty(B * S, dtype=torch.bool, device=dev) if want_mask else None
    _lib.check(lib.thd_gather(arr if fields else None, len(fields), B, S, P, _p(mask), _p(ws), ws.numel(),
                              _stream(dev)))
    return {"padding_mask": mask, "dst": dsts}


def thd_padding_mask(total_tokens: int, valid_seq_lens: torch.Tensor,
                     valid_seq_lens_padded: torch.Tensor | None = None):
    """Enqueue the layout-derived padding mask.  Returns ``(mask, info)``."""
    lib = _lib.load()
    _require_cuda("valid_seq_lens", valid_seq_lens, (torch.int64,))
    dev = valid_seq_lens.device
    if valid_seq_lens_padded is not None:
        _require_cuda("valid_seq_lens_padded", valid_seq_lens_padded, (torch.int64,), dev)
        if valid_seq_lens_padded.numel() != valid_seq_lens.numel():
            raise ValueError("valid_seq_lens_padded must match valid_seq_lens")
    n = valid_seq_lens.numel()
    mask = torch.empty(max(total_tokens, 0), dtype=torch.bool, device=dev)
    info = _new_info(dev)
    ws = _workspaces.get("thd", lib.thd_workspace_size(1, n), dev)
    _lib.check(lib.thd_padding_mask(total_tokens, _p(valid_seq_lens), _p(valid_seq_lens_padded), n, _p(mask),
                                    _p(info), _p(ws), ws.numel(), _stream(dev)))
    return mask, info


def _bins_csr(bins, dev):
    if isinstance(bins, tuple) and len(bins) == 2 and isinstance(bins[0], torch.Tensor):
        offs, mem = bins
        _require_cuda("bin_offsets", offs, (torch.int32,), dev)
        _require_cuda("bin_members", mem, (torch.int32,), dev)
        return offs, mem, int(offs.numel() - 1), int(mem.numel())
    offsets = [0]
    members = []
    for b in bins:
        members.extend(int(i) for i in b)
        offsets.append(len(members))
    offs = torch.tensor(offsets, dtype=torch.int32).to(dev)
    mem = torch.tensor(members if members else [0], dtype=torch.int32).to(dev)
    return offs, mem, len(offsets) - 1, len(members)


def pack_squeeze(src: torch.Tensor, real_lens: torch.Tensor, bins, multiple: int, capacity: int,
                 stretch_to_capacity: bool, width: int | None, pad_value: int = 0, with_output: bool = True,
                 want_mask: bool = True):
    """Enqueue the squeeze.  ``bins`` is a list of lists of row indices or a
    ``(bin_offsets, bin_members)`` pair of int32 CUDA tensors.  With
    ``with_output`` false only the metadata is produced; with ``want_mask``
    false the packed rows are produced without the padding mask.  Returns a
    dict of device tensors and the info block."""
    lib = _lib.load()
    _require_cuda("src", src)
    dev = src.device
    _require_cuda("real_lens", real_lens, (torch.int64,), dev)
    if src.dim() != 2:
        raise ValueError("src must be [N, W]")
    N, W = src.shape
    offs, mem, num_bins, M = _bins_csr(bins, dev)
    if width is None:
        width = 0
    out = torch.empty((num_bins, width), dtype=src.dtype, device=dev) if with_output else None
    mask = torch.empty((num_bins, width), dtype=torch.bool, device=dev) if with_output and want_mask else None
    cu = torch.empty(M + num_bins + 1, dtype=torch.int32, device=dev)
    cup = torch.empty(M + num_bins + 1, dtype=torch.int32, device=dev)
    info = _new_info(dev)
    ws = _workspaces.get("squeeze", lib.pack_squeeze_workspace_size(M, num_bins), dev)
    _lib.check(lib.pack_squeeze(_p(src), N, W, src.element_size(), _p(real_lens), _p(offs), _p(mem), num_bins, M,
                                multiple, capacity, 1 if stretch_to_capacity else 0, width, pad_value, _p(out),
                                _p(cu), _p(cup), _p(mask), _p(info), _p(ws), ws.numel(), _stream(dev)))
    return {"packed": out, "padding_mask": mask, "cu_seqlens": cu, "cu_seqlens_padded": cup, "info": info,
            "bin_offsets": offs, "num_bins": num_bins, "num_members": M}


# ----------------------------------------------------------------------------
# The pages' functions
# ----------------------------------------------------------------------------
@dataclass
class PackedSeqParams:
    """Packed-sequence metadata derived from a neat-packing document map.

    NeMo AutoModel packed_seq, ``PackedSeqParams``: ``cu_seqlens`` int32
    ``[num_segments + 1]`` over the flattened batch (ending at B*S),
    ``max_seqlen`` the longest segment, ``doc_ids`` passed through unchanged.
    """

    cu_seqlens: torch.Tensor
    max_seqlen: int
    doc_ids: torch.Tensor


def packed_seq_params_from_doc_ids(doc_ids: torch.Tensor) -> PackedSeqParams:
    """NeMo AutoModel packed_seq, ``packed_seq_params_from_doc_ids``."""
    cu, info = pseq_from_doc_ids(doc_ids)
    _, count, mx, _ = check_info(info, "packed_seq_params_from_doc_ids")
    return PackedSeqParams(cu_seqlens=cu[:count + 1], max_seqlen=mx, doc_ids=doc_ids)


def to_flash_attention_kwargs(params: PackedSeqParams) -> dict:
    """NeMo AutoModel packed_seq, ``to_flash_attention_kwargs``: query and key
    share one layout, so the q and k entries are the same objects."""
    return {
        "cu_seq_lens_q": params.cu_seqlens,
        "cu_seq_lens_k": params.cu_seqlens,
        "max_length_q": params.max_seqlen,
        "max_length_k": params.max_seqlen,
    }


_THD_KEYS = ("input_ids", "labels", "position_ids", "seq_lens", "seq_lens_padded")


def process_input_for_thd(batch: dict, seq_lens_padding_value: int = -1000, padding_token_id: int = 0) -> dict:
    """NeMo AutoModel v0.5 thd_utils, ``process_input_for_thd``.

    ``input_ids`` [B,S] or embeddings [B,S,H]; ``labels`` [B,S];
    ``position_ids`` [B,S] or mRoPE [n_rope,B,S]; ``seq_lens`` and
    ``seq_lens_padded`` int64 [B, num_packs].  Returns the flat THD tensors,
    ``cu_seqlens``, ``cu_seqlens_padded`` (when given), ``pad_between_seqs``
    (bool), ``max_seqlen`` (int32 scalar tensor), ``padding_mask`` (bool,
    True = padding) and every non-tensor key of the batch.  The mask comes
    from the pack layout, so ``padding_token_id`` is not consulted.
    """
    del padding_token_id  # the layout decides padding
    ids = batch["input_ids"]
    B, S = int(ids.shape[0]), int(ids.shape[1])
    fields = [(ids, 1)]
    names = ["input_ids"]
    if batch.get("labels") is not None:
        fields.append((batch["labels"], 1))
        names.append("labels")
    pos = batch.get("position_ids")
    if pos is not None:
        fields.append((pos, int(pos.shape[0]) if pos.dim() == 3 else 1))
        names.append("position_ids")
    r = thd_from_batch(batch["seq_lens"], batch.get("seq_lens_padded"), S, fields, seq_lens_padding_value, True)
    _, n, _, T = check_info(r["info"], "process_input_for_thd")
    out = {k: v for k, v in batch.items() if not isinstance(v, torch.Tensor) and k not in _THD_KEYS}
    for name, (dst, planes, row) in zip(names, r["dst"]):
        flat = dst[: planes * T * (math.prod(row) if row else 1)]
        if name == "position_ids" and planes > 1:
            out[name] = flat.view(planes, 1, T)
        else:
            out[name] = flat.view(T, *row)
    out["cu_seqlens"] = r["cu_seqlens"][: n + 1]
    if r["cu_seqlens_padded"] is not None:
        out["cu_seqlens_padded"] = r["cu_seqlens_padded"][: n + 1]
    info = r["info"]
    out["pad_between_seqs"] = bool(info[16].item())
    out["max_seqlen"] = _info_view(info)[2]
    out["padding_mask"] = r["padding_mask"][:T]
    return out


def _thd_padding_mask(total_tokens: int, valid_seq_lens: torch.Tensor,
                      valid_seq_lens_padded: torch.Tensor | None, device: torch.device | None = None) -> torch.Tensor:
    """NeMo AutoModel v0.5 thd_utils, ``_thd_padding_mask``: bool
    ``[total_tokens]``, True marks padding."""
    if device is not None and valid_seq_lens.device != torch.device(device):
        raise ValueError("valid_seq_lens must already be on the requested device")
    mask, info = thd_padding_mask(total_tokens, valid_seq_lens, valid_seq_lens_padded)
    check_info(info, "_thd_padding_mask")
    return mask


def squeeze_bins(input_ids: torch.Tensor, input_lengths: torch.Tensor, bins, multiple: int, capacity: int,
                 stretch_to_capacity: bool = False, width: int | None = None, pad_value: int = 0) -> dict:
    """The trainer-side squeeze of "Who packs the sequences".

    Concatenates the sources of each bin end to end, each padded to
    ``multiple``.  ``width`` defaults to the pack capacity when stretching
    (loader-style rows) and to the widest bin otherwise (trainer-style rows).
    Returns ``packed_input_ids`` [num_bins, width], ``padding_mask``
    (True = padding), and per-bin lists ``cu_seqlens`` / ``cu_seqlens_padded``
    (views into the flat arrays ``cu_seqlens_flat`` / ``cu_seqlens_padded_flat``).
    """
    _require_cuda("input_ids", input_ids)
    offs, mem, _, _ = _bins_csr(bins, input_ids.device)
    bins = (offs, mem)
    if width is None and stretch_to_capacity:
        width = capacity
    if width is None:
        meta = pack_squeeze(input_ids, input_lengths, bins, multiple, capacity, False, None, pad_value,
                            with_output=False)
        _, _, _, width = check_info(meta["info"], "squeeze_bins")
    r = pack_squeeze(input_ids, input_lengths, bins, multiple, capacity, stretch_to_capacity, width, pad_value)
    check_info(r["info"], "squeeze_bins")
    offs = r["bin_offsets"].tolist()
    cu, cup = r["cu_seqlens"], r["cu_seqlens_padded"]
    return {
        "packed_input_ids": r["packed"],
        "padding_mask": r["padding_mask"],
        "cu_seqlens": [cu[offs[b] + b: offs[b + 1] + b + 1] for b in range(r["num_bins"])],
        "cu_seqlens_padded": [cup[offs[b] + b: offs[b + 1] + b + 1] for b in range(r["num_bins"])],
        "cu_seqlens_flat": cu[: r["num_members"] + r["num_bins"]],
        "cu_seqlens_padded_flat": cup[: r["num_members"] + r["num_bins"]],
    }


# ----------------------------------------------------------------------------
# chunked THD, value mask, bin packing, doc_ids bridge (C entry points)
# ----------------------------------------------------------------------------
def thd_chunks_from_batch(seq_lens: torch.Tensor, seq_lens_padded: torch.Tensor | None, S: int, num_chunks: int,
                          fields=(), pad_value: int = -1000, absorb_trailing_pad: bool = True, want_mask: bool = True):
    """Enqueue the chunked conversion.  Returns device buffers sized for the
    worst case, ``infos`` (num_chunks x 16 bytes) and ``pad_between``
    (num_chunks bytes)."""
    lib = _lib.load()
    _require_cuda("seq_lens", seq_lens, (torch.int64,))
    dev = seq_lens.device
    if seq_lens_padded is not None:
        _require_cuda("seq_lens_padded", seq_lens_padded, (torch.int64,), dev)
        if seq_lens_padded.shape != seq_lens.shape:
            raise ValueError("seq_lens_padded must have the shape of seq_lens")
    B, P = seq_lens.shape
    if num_chunks < 1 or B % num_chunks:
        raise ValueError("num_chunks must evenly divide the batch size")
    Bc = B // num_chunks
    arr, dsts = _fields(fields, B, S, dev)
    width = Bc * P + 1
    cu = torch.empty((num_chunks, width), dtype=torch.int32, device=dev)
    cup = torch.empty((num_chunks, width), dtype=torch.int32, device=dev) if seq_lens_padded is not None else None
    mask = torch.empty(B * S, dtype=torch.bool, device=dev) if want_mask else None
    infos = torch.empty((num_chunks, 4), dtype=torch.int32, device=dev)
    pbs = torch.empty(num_chunks, dtype=torch.uint8, device=dev)
    ws = _workspaces.get("thd", lib.thd_workspace_size(Bc, P), dev)
    _lib.check(lib.thd_chunks_from_batch(_p(seq_lens), _p(seq_lens_padded), B, S, P, num_chunks, pad_value,
                                         1 if absorb_trailing_pad else 0, arr if fields else None, len(fields),
                                         _p(cu), _p(cup), _p(mask), _p(pbs), _p(infos), _p(ws), ws.numel(),
                                         _stream(dev)))
    return {"cu_seqlens": cu, "cu_seqlens_padded": cup, "padding_mask": mask, "dst": dsts, "infos": infos,
            "pad_between": pbs}


def thd_mask_from_token_ids(input_ids: torch.Tensor, padding_token_id: int):
    """Enqueue the value-compare mask.  Returns ``(mask, info)``."""
    lib = _lib.load()
    _require_cuda("input_ids", input_ids, (torch.int32, torch.int64))
    dev = input_ids.device
    n = input_ids.numel()
    mask = torch.empty(n, dtype=torch.bool, device=dev)
    info = _new_info(dev)
    ws = _workspaces.get("token_mask", lib.thd_mask_from_token_ids_workspace_size(n), dev)
    _lib.check(lib.thd_mask_from_token_ids(_p(input_ids), input_ids.element_size(), n, int(padding_token_id),
                                           _p(mask), _p(info), _p(ws), ws.numel(), _stream(dev)))
    return mask.view(input_ids.shape), info


def pack_ffd(lens: torch.Tensor, capacity: int, multiple: int = 1):
    """Enqueue first-fit-decreasing.  Returns ``(bin_offsets [n+1],
    bin_members [n], info)``; the first ``info.count + 1`` offsets are valid."""
    lib = _lib.load()
    _require_cuda("lens", lens, (torch.int64,))
    dev = lens.device
    n = lens.numel()
    offs = torch.empty(n + 1, dtype=torch.int32, device=dev)
    mem = torch.empty(max(n, 1), dtype=torch.int32, device=dev)
    info = _new_info(dev)
    _lib.check(lib.pack_ffd(_p(lens), n, multiple, capacity, _p(offs), _p(mem), _p(info), _stream(dev)))
    return offs, mem[:n], info


def pseq_doc_ids_to_lengths(doc_ids: torch.Tensor, num_packs: int, pad_value: int = -1000,
                            with_positions: bool = True):
    """Enqueue the doc_ids -> pack lengths bridge.  Returns ``(seq_lens,
    seq_lens_padded, position_ids or None, info)``."""
    lib = _lib.load()
    _require_cuda("doc_ids", doc_ids, (torch.int32, torch.int64))
    if doc_ids.dim() != 2:
        raise ValueError("doc_ids must be [batch, sequence]")
    dev = doc_ids.device
    B, S = doc_ids.shape
    real = torch.empty((B, num_packs), dtype=torch.int64, device=dev)
    padded = torch.empty((B, num_packs), dtype=torch.int64, device=dev)
    pos = torch.empty((B, S), dtype=torch.int64, device=dev) if with_positions else None
    info = _new_info(dev)
    ws = _workspaces.get("bridge", lib.pseq_doc_ids_to_lengths_workspace_size(B, S), dev)
    _lib.check(lib.pseq_doc_ids_to_lengths(_p(doc_ids), doc_ids.element_size(), B, S, num_packs, pad_value, _p(real),
                                           _p(padded), _p(pos), _p(info), _p(ws), ws.numel(), _stream(dev)))
    return real, padded, pos, info


# ----------------------------------------------------------------------------
# the pages' functions for those rows
# ----------------------------------------------------------------------------
def split_batch_into_thd_chunks(batch: dict, num_chunks: int, seq_lens_padding_value: int = -1000,
                                padding_token_id: int = 0) -> dict:
    """NeMo AutoModel v0.5 thd_utils, ``split_batch_into_thd_chunks``.

    Splits the batch along its rows into ``num_chunks`` chunks, converts each
    as ``process_input_for_thd`` does and stacks the results on a new leading
    axis; ``cu_seqlens`` / ``cu_seqlens_padded`` rows are padded with
    ``seq_lens_padding_value``.  ``max_seqlen`` becomes an int32 tensor
    [num_chunks] and ``pad_between_seqs`` a bool tensor [num_chunks].
    Chunks whose streams differ in length cannot be stacked: ValueError.
    The stacked tensors are views of the library's chunked buffers, in which
    chunk c starts at a fixed stride of (B / num_chunks) * S rows; they are
    contiguous when every chunk's stream fills its rows (T == B/num_chunks*S).
    """
    if num_chunks <= 1:
        return process_input_for_thd(batch, seq_lens_padding_value, padding_token_id)
    ids = batch["input_ids"]
    B, S = int(ids.shape[0]), int(ids.shape[1])
    fields = [(ids, 1)]
    names = ["input_ids"]
    if batch.get("labels") is not None:
        fields.append((batch["labels"], 1))
        names.append("labels")
    pos = batch.get("position_ids")
    if pos is not None:
        fields.append((pos, int(pos.shape[0]) if pos.dim() == 3 else 1))
        names.append("position_ids")
    r = thd_chunks_from_batch(batch["seq_lens"], batch.get("seq_lens_padded"), S, num_chunks, fields,
                              seq_lens_padding_value, True)
    infos = r["infos"].tolist()
    for c, (st, _, _, _) in enumerate(infos):
        if st != _lib.PSEQ_OK:
            name = _lib.STATUS_NAMES.get(st, str(st))
            raise (ValueError if st in (_lib.PSEQ_ERR_VALUE, _lib.PSEQ_ERR_CAPACITY) else RuntimeError)(
                f"split_batch_into_thd_chunks: chunk {c}: device reported {name}")
    totals = {t for _, _, _, t in infos}
    if len(totals) != 1:
        raise ValueError(f"split_batch_into_thd_chunks: chunk streams have different lengths {sorted(totals)} "
                         "and cannot be stacked")
    T = totals.pop()
    Sc = B // num_chunks * S  # the library writes chunk c's stream and mask at a fixed stride of Sc rows
    width = max(n for _, n, _, _ in infos) + 1
    out = {k: v for k, v in batch.items() if not isinstance(v, torch.Tensor) and k not in _THD_KEYS}
    for name, (dst, planes, row) in zip(names, r["dst"]):
        # views of the chunks' streams, stacked on a leading axis (contiguous when T == Sc)
        per_chunk = dst.view(num_chunks, planes * Sc, *row)[:, : planes * T]
        if name == "position_ids" and planes > 1:
            out[name] = per_chunk.view(num_chunks, planes, 1, T)
        else:
            out[name] = per_chunk
    out["cu_seqlens"] = r["cu_seqlens"][:, :width]
    if r["cu_seqlens_padded"] is not None:
        out["cu_seqlens_padded"] = r["cu_seqlens_padded"][:, :width]
    out["pad_between_seqs"] = r["pad_between"].view(torch.bool)
    out["max_seqlen"] = r["infos"][:, 2]
    out["padding_mask"] = r["padding_mask"].view(num_chunks, Sc)[:, :T]
    return out


def thd_padding_mask_from_token_ids(input_ids: torch.Tensor, padding_token_id: int) -> torch.Tensor:
    """NeMo AutoModel v0.5 thd_utils, ``thd_padding_mask_from_token_ids``:
    bool mask (True = padding) by value; ValueError when the pad id also
    occurs as content (anywhere before the suffix of pad tokens)."""
    mask, info = thd_mask_from_token_ids(input_ids, padding_token_id)
    st = _info_view(info).tolist()[0]
    if st != _lib.PSEQ_OK:
        raise ValueError(f"padding_token_id {padding_token_id} also occurs as content")
    return mask


def first_fit_decreasing(lens: torch.Tensor, capacity: int, multiple: int = 1):
    """First-fit-decreasing bins ("Who packs the sequences": get_packer, by
    token budget).  Returns ``(bin_offsets, bin_members)`` int32 CUDA tensors,
    ready for ``pack_squeeze``."""
    offs, mem, info = pack_ffd(lens, capacity, multiple)
    _, nb, _, _ = check_info(info, "first_fit_decreasing")
    return offs[: nb + 1], mem


def doc_ids_to_seq_lens(doc_ids: torch.Tensor, num_packs: int | None = None, pad_value: int = -1000) -> dict:
    """From a neat-packing document map to ``seq_lens``, ``seq_lens_padded``
    [B, num_packs] and ``position_ids`` [B, S] for ``process_input_for_thd``.
    ``num_packs`` defaults to the most sequences any row holds."""
    if num_packs is None:
        # first pass sizes the table: the most sequences any row holds
        S = int(doc_ids.shape[1]) if doc_ids.dim() == 2 else 0
        _, _, _, info = pseq_doc_ids_to_lengths(doc_ids, S, pad_value, with_positions=False)
        _, num_packs, _, _ = check_info(info, "doc_ids_to_seq_lens")
    real, padded, pos, info = pseq_doc_ids_to_lengths(doc_ids, num_packs, pad_value)
    check_info(info, "doc_ids_to_seq_lens")
    return {"seq_lens": real, "seq_lens_padded": padded, "position_ids": pos}

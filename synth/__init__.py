"""Seeded synthetic inputs for the packed-sequence metadata path.

This module builds inputs only.  It holds none of the method's arithmetic
(no segmentation, filtering, cumulative sums, gathers or masks): the CUDA
path and the CPU oracle both consume what it returns, and neither is
imported here.  Every array is drawn from ``numpy.random.default_rng(seed)``.

Workloads (shapes and distributions of packed supervised fine-tuning batches):

* ``doc_map_small``   doc_ids int32 [4, 2048]: documents of length
  uniform[16, 512] numbered 1.. per row, then a tail padding run of
  uniform[0, 256] zeros; with a matching THD batch of int64 ids, labels and
  per-document positions.
* ``thd_ids``         B=8, S=8192, 64 pack slots: lognormal(6, 1) lengths
  clipped to the row, padded to a multiple of 64, unused slots -1000; int64
  ids and labels, mRoPE positions [3, 8, 8192].
* ``thd_embeddings``  bf16 hidden [4, 8192, 4096] ~ N(0, 1) with the same
  length distribution as ``thd_ids``; ``thd_embeddings_ragged`` drops each
  row's last sequence, so rows end short and sequences move.
* ``squeeze``         256 sources in an int64 rectangle [256, 4096] with real
  lengths lognormal(6.5, 0.8) clipped to [1, 4096], multiple 64, bins by
  first-fit-decreasing at capacity 32768, output width 32768, stretched.
* ``doc_map_stress``  doc_ids int32 [64, 32768]: runs of geometric length
  (mean 8, at most 4096), each a new document with probability 0.9 and a
  zero run otherwise, then a tail zero run of uniform[0, 256].
"""
from __future__ import annotations

import numpy as np

FILLER = -1000
VOCAB = 32000


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# doc_ids maps
# --------------------------------------------------------------------------
def doc_map_small(seed: int = 0, B: int = 4, S: int = 2048) -> dict:
    """Neat-packing map plus its THD companion batch (see module docstring)."""
    rng = _rng(seed)
    doc_ids = np.zeros((B, S), np.int32)
    position_ids = np.zeros((B, S), np.int64)
    row_docs = []
    row_tails = []
    for b in range(B):
        tail = int(rng.integers(0, 256, endpoint=True))
        tail = min(tail, S)
        fill = S - tail
        lengths = []
        pos = 0
        while pos < fill:
            L = int(rng.integers(16, 512, endpoint=True))
            L = min(L, fill - pos)
            doc_ids[b, pos:pos + L] = len(lengths) + 1
            position_ids[b, pos:pos + L] = np.arange(L)
            lengths.append(L)
            pos += L
        row_docs.append(lengths)
        row_tails.append(tail)
    P = max(1, max(len(d) for d in row_docs))
    seq_lens = np.full((B, P), FILLER, np.int64)
    seq_lens_padded = np.full((B, P), FILLER, np.int64)
    for b, lengths in enumerate(row_docs):
        for c, L in enumerate(lengths):
            seq_lens[b, c] = L
            seq_lens_padded[b, c] = L
        if lengths:
            seq_lens_padded[b, len(lengths) - 1] += row_tails[b]
        elif row_tails[b]:
            # a row that is all padding carries one empty sequence owning it
            seq_lens[b, 0] = 0
            seq_lens_padded[b, 0] = row_tails[b]
    input_ids = rng.integers(0, VOCAB, size=(B, S), dtype=np.int64)
    labels = rng.integers(0, VOCAB, size=(B, S), dtype=np.int64)
    return {
        "doc_ids": doc_ids,
        "input_ids": input_ids,
        "labels": labels,
        "position_ids": position_ids,
        "seq_lens": seq_lens,
        "seq_lens_padded": seq_lens_padded,
    }


def doc_map_stress(seed: int = 0, B: int = 64, S: int = 32768, p_zero: float = 0.1,
                   mean_len: int = 8, max_len: int = 4096, max_tail: int = 256) -> np.ndarray:
    """Many short documents with zero runs inside and at the tail of each row."""
    rng = _rng(seed)
    doc_ids = np.zeros((B, S), np.int32)
    for b in range(B):
        tail = min(int(rng.integers(0, max_tail, endpoint=True)), S)
        fill = S - tail
        pos = 0
        next_id = 1
        while pos < fill:
            k = 4096
            lengths = np.minimum(rng.geometric(1.0 / mean_len, size=k), max_len)
            is_zero = rng.random(k) < p_zero
            for L, z in zip(lengths.tolist(), is_zero.tolist()):
                if pos >= fill:
                    break
                L = min(L, fill - pos)
                if not z:
                    doc_ids[b, pos:pos + L] = next_id
                    next_id += 1
                pos += L
    return doc_ids


def random_doc_ids(rng: np.random.Generator, B: int, S: int, kind: str = "runs",
                   dtype=np.int32) -> np.ndarray:
    """Small random maps for parity tests.

    kinds: ``runs`` (geometric runs, ids 0..3 reused, so equal ids recur after
    a change), ``iid`` (every token uniform in {0,1,2}), ``zeros`` (all
    padding), ``const`` (one id everywhere), ``alternating`` (1,2,1,2..),
    ``long`` (runs longer than a row).
    """
    if kind == "iid":
        return rng.integers(0, 3, size=(B, S)).astype(dtype)
    if kind == "zeros":
        return np.zeros((B, S), dtype)
    if kind == "const":
        return np.full((B, S), 7, dtype)
    if kind == "alternating":
        return (np.arange(B * S).reshape(B, S) % 2 + 1).astype(dtype)
    mean = {"runs": 6, "long": max(2, 3 * S)}[kind]
    flat = np.zeros(B * S, np.int64)
    pos = 0
    while pos < B * S:
        L = int(rng.geometric(1.0 / mean))
        flat[pos:pos + L] = int(rng.integers(0, 4))
        pos += L
    return flat.reshape(B, S).astype(dtype)


# --------------------------------------------------------------------------
# BSHD batches with pack lengths
# --------------------------------------------------------------------------
def _ceil_to(x: int, m: int) -> int:
    return -(-x // m) * m


def pack_lengths(rng: np.random.Generator, B: int, S: int, P: int, mu: float = 6.0,
                 sigma: float = 1.0, multiple: int = 64):
    """Per row, draw lengths until the row is full or the P slots are used.

    ``real = max(1, round(lognormal(mu, sigma)))`` clipped to what is left of
    the row; ``padded`` is ``real`` rounded up to ``multiple``, clipped to
    what is left.  Unused slots hold -1000 in both arrays.
    """
    seq_lens = np.full((B, P), FILLER, np.int64)
    seq_lens_padded = np.full((B, P), FILLER, np.int64)
    for b in range(B):
        rem = S
        c = 0
        while c < P and rem > 0:
            L = max(1, int(round(rng.lognormal(mu, sigma))))
            L = min(L, rem)
            Lp = min(_ceil_to(L, multiple), rem)
            seq_lens[b, c] = L
            seq_lens_padded[b, c] = Lp
            rem -= Lp
            c += 1
    return seq_lens, seq_lens_padded


def _positions(seq_lens_padded: np.ndarray, seq_lens: np.ndarray, S: int) -> np.ndarray:
    """Position within each sequence for real tokens, 0 on padding slots."""
    B, P = seq_lens.shape
    pos = np.zeros((B, S), np.int64)
    for b in range(B):
        o = 0
        for c in range(P):
            if seq_lens[b, c] == FILLER:
                continue
            pos[b, o:o + seq_lens[b, c]] = np.arange(seq_lens[b, c])
            o += int(seq_lens_padded[b, c])
    return pos


def thd_ids(seed: int = 0, B: int = 8, S: int = 8192, P: int = 64, n_rope: int = 3) -> dict:
    """process_input_for_thd batch with int64 ids/labels and mRoPE positions."""
    rng = _rng(seed)
    seq_lens, seq_lens_padded = pack_lengths(rng, B, S, P)
    input_ids = rng.integers(0, VOCAB, size=(B, S), dtype=np.int64)
    labels = rng.integers(0, VOCAB, size=(B, S), dtype=np.int64)
    pos = np.zeros((n_rope, B, S), np.int64)
    pos[0] = _positions(seq_lens_padded, seq_lens, S)
    if n_rope > 1:
        pos[1:] = rng.integers(0, 64, size=(n_rope - 1, B, S), dtype=np.int64)
    return {
        "input_ids": input_ids,
        "labels": labels,
        "position_ids": pos,
        "seq_lens": seq_lens,
        "seq_lens_padded": seq_lens_padded,
    }


def thd_embeddings(seed: int = 0, B: int = 4, S: int = 8192, H: int = 4096, P: int = 64) -> dict:
    """bf16 hidden states [B, S, H] ~ N(0, 1) with thd_ids-style lengths.

    ``hidden`` is returned as a CPU ``torch.bfloat16`` tensor (numpy has no
    bfloat16); the values are only ever copied, never computed on.
    """
    import torch

    rng = _rng(seed + 7919)  # distinct stream from thd_ids at the same seed
    seq_lens, seq_lens_padded = pack_lengths(rng, B, S, P)
    x = rng.standard_normal(size=(B, S, H), dtype=np.float32)
    hidden = torch.from_numpy(x).to(torch.bfloat16)
    return {"hidden": hidden, "seq_lens": seq_lens, "seq_lens_padded": seq_lens_padded}


def thd_embeddings_ragged(seed: int = 0, B: int = 4, S: int = 8192, H: int = 4096, P: int = 64) -> dict:
    """``thd_embeddings`` with every row ending short: each row's last kept
    sequence is set to -1000 in both length arrays (the slots stay in the
    hidden tensor but are no longer part of the batch), so the stream is
    shorter than B*S and every row after the first lands in the stream at a
    different offset than it has in the batch."""
    c = thd_embeddings(seed, B, S, H, P)
    for b in range(B):
        kept = np.nonzero(c["seq_lens"][b] != FILLER)[0]
        if kept.size > 1:
            c["seq_lens"][b, kept[-1]] = FILLER
            c["seq_lens_padded"][b, kept[-1]] = FILLER
    return c


def random_thd(rng: np.random.Generator, B: int, S: int, P: int, multiple: int = 4,
               interleave_filler: bool = True, fill_rows: bool = False,
               with_zero_lengths: bool = True):
    """Small random seq_lens / seq_lens_padded pairs for parity tests.

    Rows may end short of S, filler entries may sit between kept ones, and
    zero-length sequences may occur.  ``fill_rows`` makes every row's padded
    lengths sum to exactly S.
    """
    seq_lens = np.full((B, P), FILLER, np.int64)
    seq_lens_padded = np.full((B, P), FILLER, np.int64)
    for b in range(B):
        rem = S
        for c in range(P):
            if rem <= 0:
                break
            if interleave_filler and rng.random() < 0.2:
                continue
            lo = 0 if with_zero_lengths else 1
            L = int(rng.integers(lo, max(lo, min(rem, 2 * multiple + 3)) + 1))
            L = min(L, rem)
            Lp = min(_ceil_to(L, multiple) + int(rng.integers(0, 2)) * multiple, rem)
            Lp = max(Lp, L)
            seq_lens[b, c] = L
            seq_lens_padded[b, c] = Lp
            rem -= Lp
        if fill_rows and rem > 0:
            kept = np.nonzero(seq_lens[b] != FILLER)[0]
            if kept.size:
                seq_lens_padded[b, kept[-1]] += rem
            else:
                seq_lens[b, 0] = 0
                seq_lens_padded[b, 0] = rem
    return seq_lens, seq_lens_padded


# --------------------------------------------------------------------------
# trainer-side squeeze
# --------------------------------------------------------------------------
def first_fit_decreasing(sizes, capacity: int):
    """Bin assignment used as INPUT by the squeeze workload.

    Sort by size descending (ties by index), put each item in the first bin
    with room, open a new bin when none has room.  Returns a list of bins,
    each a list of source indices in placement order.
    """
    order = sorted(range(len(sizes)), key=lambda i: (-int(sizes[i]), i))
    bins, room = [], []
    for i in order:
        s = int(sizes[i])
        for k in range(len(bins)):
            if room[k] >= s:
                bins[k].append(i)
                room[k] -= s
                break
        else:
            bins.append([i])
            room.append(capacity - s)
    return bins


def squeeze(seed: int = 0, N: int = 256, W: int = 4096, multiple: int = 64,
            capacity: int = 32768, mu: float = 6.5, sigma: float = 0.8) -> dict:
    """Padded rectangle, real lengths and an FFD bin assignment (as CSR)."""
    rng = _rng(seed)
    real = np.clip(np.round(rng.lognormal(mu, sigma, size=N)), 1, W).astype(np.int64)
    src = rng.integers(0, VOCAB, size=(N, W), dtype=np.int64)
    src[np.arange(W)[None, :] >= real[:, None]] = 0
    padded_sizes = [_ceil_to(int(r), multiple) for r in real]
    bins = first_fit_decreasing(padded_sizes, capacity)
    offsets = np.zeros(len(bins) + 1, np.int32)
    members = []
    for b, m in enumerate(bins):
        members.extend(m)
        offsets[b + 1] = len(members)
    return {
        "src": src,
        "real_lens": real,
        "bin_offsets": offsets,
        "bin_members": np.asarray(members, np.int32),
        "bins": bins,
        "multiple": multiple,
        "capacity": capacity,
        "width": capacity,
        "stretch": True,
        "pad_value": 0,
    }


def random_squeeze(rng: np.random.Generator, N: int, W: int, num_bins: int,
                   elem_dtype=np.int64, allow_zero: bool = True) -> dict:
    """Small random squeeze problems: random lengths, random bin membership."""
    lo = 0 if allow_zero else 1
    real = rng.integers(lo, W + 1, size=N).astype(np.int64)
    if np.issubdtype(elem_dtype, np.integer):
        info = np.iinfo(elem_dtype)
        src = rng.integers(max(info.min, -30000), min(info.max, 30000), size=(N, W)).astype(elem_dtype)
    else:
        src = rng.standard_normal((N, W)).astype(elem_dtype)
    perm = rng.permutation(N)
    cuts = np.sort(rng.choice(np.arange(1, N), size=min(num_bins - 1, N - 1), replace=False)) if N > 1 else []
    groups = np.split(perm, cuts)
    bins = [g.tolist() for g in groups if len(g)]
    offsets = np.zeros(len(bins) + 1, np.int32)
    members = []
    for b, m in enumerate(bins):
        members.extend(m)
        offsets[b + 1] = len(members)
    return {"src": src, "real_lens": real, "bin_offsets": offsets,
            "bin_members": np.asarray(members, np.int32), "bins": bins}

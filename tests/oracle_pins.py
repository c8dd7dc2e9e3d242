"""Checks that pin the CPU oracle to something other than itself.

Each ``pin_*`` function takes an oracle library handle and raises
``AssertionError`` when the oracle disagrees with:

* a worked example printed on the pages (fixtures under ``tests/golden/``),
* a closed form or invariant the pages state,
* a library routine the operation reduces to (run-length encoding through
  ``torch.unique_consecutive``, flattening through ``reshape``),
* brute force over every tiny input.

``test_oracle_pins.py`` runs them against the real oracle;
``test_oracle_mutants.py`` runs them against copies of the oracle with a
planted mistake and requires that some pin fails for every mistake.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# O1 packed_seq_params_from_doc_ids
# --------------------------------------------------------------------------
def _rle_reference(doc_ids: np.ndarray):
    """cu_seqlens by run-length encoding of the key (row, doc) in torch."""
    B, S = doc_ids.shape
    if B * S == 0:
        return np.zeros(1, np.int32), 0
    rows = np.repeat(np.arange(B, dtype=np.int64), S)
    docs = doc_ids.reshape(-1).astype(np.int64)
    # a key that is unique per (row, doc) pair; docs fit in 40 bits here
    key = torch.from_numpy(rows * (1 << 40) + (docs + (1 << 39)))
    _, counts = torch.unique_consecutive(key, return_counts=True)
    cu = np.concatenate([[0], np.cumsum(counts.numpy())]).astype(np.int32)
    return cu, int(counts.max())


def pin_doc_ids_page_example(lib):
    g = golden("packed_seq_doc_ids_example.json")
    cu, mx = oracle.from_doc_ids(np.asarray(g["doc_ids"], np.int32), lib=lib)
    assert cu.tolist() == g["cu_seqlens"], cu
    assert mx == g["max_seqlen"], mx


def pin_doc_ids_brute_force(lib, max_tokens: int = 7):
    """Every map in {0,1,2}^(B*S) with B*S <= max_tokens, every B x S."""
    for n in range(1, max_tokens + 1):
        shapes = [(B, n // B) for B in range(1, n + 1) if n % B == 0]
        for vals in itertools.product((0, 1, 2), repeat=n):
            flat = np.asarray(vals, np.int32)
            for B, S in shapes:
                d = flat.reshape(B, S)
                cu, mx = oracle.from_doc_ids(d, lib=lib)
                ref_cu, ref_mx = _rle_reference(d)
                assert np.array_equal(cu, ref_cu), (d.tolist(), cu, ref_cu)
                assert mx == ref_mx, (d.tolist(), mx, ref_mx)


def pin_doc_ids_invariants(lib, seeds=range(6)):
    """cu[0]=0, strictly increasing, ends at B*S, every row start present,
    one id per segment, adjacent same-row segments differ; RLE agreement."""
    for seed in seeds:
        rng = np.random.default_rng(seed)
        for kind in ("runs", "iid", "zeros", "const", "alternating", "long"):
            B, S = int(rng.integers(1, 6)), int(rng.integers(1, 40))
            for dtype in (np.int32, np.int64):
                d = synth.random_doc_ids(rng, B, S, kind, dtype)
                cu, mx = oracle.from_doc_ids(d, lib=lib)
                flat = d.reshape(-1)
                assert cu[0] == 0 and cu[-1] == B * S
                assert np.all(np.diff(cu) > 0)
                assert set(range(0, B * S, S)) <= set(cu.tolist())
                for k in range(len(cu) - 1):
                    seg = flat[cu[k]:cu[k + 1]]
                    assert np.all(seg == seg[0])
                    assert cu[k] // S == (cu[k + 1] - 1) // S  # no segment crosses a row
                    if k + 1 < len(cu) - 1 and cu[k + 1] % S != 0:
                        assert flat[cu[k + 1]] != flat[cu[k + 1] - 1]
                assert mx == int(np.diff(cu).max())
                ref_cu, ref_mx = _rle_reference(d)
                assert np.array_equal(cu, ref_cu) and mx == ref_mx


def pin_doc_ids_empty(lib):
    for shape in ((0, 5), (3, 0), (0, 0)):
        cu, mx = oracle.from_doc_ids(np.zeros(shape, np.int32), lib=lib)
        assert cu.tolist() == [0] and mx == 0


# --------------------------------------------------------------------------
# O2-O4 process_input_for_thd and _thd_padding_mask
# --------------------------------------------------------------------------
def pin_thd_page_example(lib):
    g = golden("thd_utils_process_input_example.json")
    batch = {k: np.asarray(v, np.int64) for k, v in g["batch"].items()}
    out = oracle.process_input_for_thd(batch, lib=lib)
    e = g["expected"]
    for k in ("input_ids", "labels", "position_ids", "cu_seqlens", "cu_seqlens_padded"):
        assert np.asarray(out[k]).tolist() == e[k], (k, out[k])
    assert out["max_seqlen"] == e["max_seqlen"]
    assert out["padding_mask"].tolist() == e["padding_mask"]
    assert out["pad_between_seqs"] == e["pad_between_seqs"]
    assert out["total_tokens"] == e["total_tokens"]


def _row_prefix_concat(x: np.ndarray, row_used: np.ndarray) -> np.ndarray:
    """Concatenation over rows of each row's first row_used[b] slots."""
    return np.concatenate([x[b, :row_used[b]] for b in range(x.shape[0])], axis=0)


def pin_thd_closed_forms(lib, seeds=range(12)):
    """On random layouts (filler between kept entries, short rows, zero
    lengths): the stream is the concatenation of each row's used prefix;
    the mask has T - sum(real) set bits, marking exactly the slots past each
    sequence's real tokens; cu differences are the kept lengths in row-major
    order; max_seqlen equals the largest final difference."""
    for seed in seeds:
        rng = np.random.default_rng(100 + seed)
        B, S, P = int(rng.integers(1, 5)), int(rng.integers(1, 50)), int(rng.integers(1, 7))
        real, padded = synth.random_thd(rng, B, S, P, multiple=int(rng.integers(1, 5)),
                                        fill_rows=bool(seed % 2))
        ids = rng.integers(0, 1000, size=(B, S)).astype(np.int64)
        pos3 = rng.integers(0, 1000, size=(3, B, S)).astype(np.int64)
        hid = rng.integers(-5000, 5000, size=(B, S, 3)).astype(np.int16)
        for absorb in (True, False):
            out = oracle.process_input_for_thd(
                {"input_ids": ids, "labels": ids + 1, "position_ids": pos3,
                 "seq_lens": real, "seq_lens_padded": padded}, absorb=absorb, lib=lib)
            keep = real != -1000
            kept_real = real[keep]
            kept_padded = padded[keep]
            row_used = np.where(keep, padded, 0).sum(axis=1)
            T = int(row_used.sum())
            assert out["total_tokens"] == T
            assert np.array_equal(out["input_ids"], _row_prefix_concat(ids, row_used))
            assert np.array_equal(out["labels"], _row_prefix_concat(ids + 1, row_used))
            assert out["position_ids"].shape == (3, 1, T)
            for p in range(3):
                assert np.array_equal(out["position_ids"][p, 0], _row_prefix_concat(pos3[p], row_used))
            cu, cup = out["cu_seqlens"], out["cu_seqlens_padded"]
            assert np.array_equal(np.diff(cup), kept_padded)
            n = kept_real.size
            pad_inside = n > 0 and bool(np.any(kept_real[:-1] != kept_padded[:-1]))
            absorbed = absorb and n > 0 and not pad_inside
            if absorbed:
                assert np.array_equal(cu, cup)
                assert not out["pad_between_seqs"]
            else:
                assert np.array_equal(np.diff(cu), kept_real)
                assert out["pad_between_seqs"] == bool(np.any(kept_real != kept_padded))
            assert out["max_seqlen"] == (int(np.diff(cu).max()) if n else 0)
            mask = out["padding_mask"]
            assert int(mask.sum()) == T - int(kept_real.sum())
            want = np.concatenate([np.r_[np.zeros(r, bool), np.ones(q - r, bool)]
                                   for r, q in zip(kept_real, kept_padded)] or [np.zeros(0, bool)])
            assert np.array_equal(mask, want)
            emb = oracle.thd_gather(hid, oracle.thd_meta(real, padded, S, lib=lib), B, S, lib=lib)
            assert np.array_equal(emb, _row_prefix_concat(hid, row_used))


def pin_thd_full_rows_is_reshape(lib, seeds=range(4)):
    """When every row's padded lengths fill the row, the stream is the
    row-major flattening (the page's 'collapsed to 1D' / 'Reshaped')."""
    for seed in seeds:
        rng = np.random.default_rng(200 + seed)
        B, S, P = 3, 24, 6
        real, padded = synth.random_thd(rng, B, S, P, multiple=4, fill_rows=True)
        x = rng.integers(0, 1 << 40, size=(B, S)).astype(np.int64)
        out = oracle.process_input_for_thd({"input_ids": x, "seq_lens": real, "seq_lens_padded": padded}, lib=lib)
        assert np.array_equal(out["input_ids"], x.reshape(-1))
        assert out["total_tokens"] == B * S


def pin_thd_absorption(lib):
    """Trailing-only pad is absorbed (cu == cu_padded, pad_between False);
    inner pad is not (the page's Example keeps [0,3,5,11])."""
    S = 10
    real = np.array([[2, 3, 1]], np.int64)
    padded = np.array([[2, 3, 5]], np.int64)
    m = oracle.thd_meta(real, padded, S, lib=lib)
    assert m["cu_seqlens"].tolist() == [0, 2, 5, 10]
    assert m["cu_seqlens_padded"].tolist() == [0, 2, 5, 10]
    assert m["pad_between_seqs"] is False
    assert m["max_seqlen"] == 5
    m = oracle.thd_meta(real, padded, S, absorb=False, lib=lib)
    assert m["cu_seqlens"].tolist() == [0, 2, 5, 6]
    assert m["pad_between_seqs"] is True
    assert m["max_seqlen"] == 3
    inner = oracle.thd_meta(np.array([[1, 3, 1]]), np.array([[2, 3, 5]]), S, lib=lib)
    assert inner["cu_seqlens"].tolist() == [0, 1, 4, 5]
    assert inner["pad_between_seqs"] is True
    # no padded lengths: padded := real, nothing to absorb or compare
    none = oracle.thd_meta(real, None, S, lib=lib)
    assert none["cu_seqlens"].tolist() == [0, 2, 5, 6]
    assert none["total_tokens"] == 6 and none["pad_between_seqs"] is False


def pin_thd_empty_and_filler_only(lib):
    m = oracle.thd_meta(np.full((2, 3), -1000, np.int64), np.full((2, 3), -1000, np.int64), 8, lib=lib)
    assert m["cu_seqlens"].tolist() == [0] and m["cu_seqlens_padded"].tolist() == [0]
    assert m["total_tokens"] == 0 and m["max_seqlen"] == 0 and m["pad_between_seqs"] is False
    m = oracle.thd_meta(np.zeros((0, 3), np.int64), np.zeros((0, 3), np.int64), 8, lib=lib)
    assert m["cu_seqlens"].tolist() == [0] and m["total_tokens"] == 0


def pin_thd_errors(lib):
    S = 8
    bad = [
        (np.array([[3, -1000]]), np.array([[3, 4]])),   # filler in one array only
        (np.array([[3, 2]]), np.array([[2, 2]])),       # padded < real
        (np.array([[-2, 2]]), np.array([[-2, 2]])),     # negative length
        (np.array([[5, 3]]), np.array([[5, 4]])),       # row overflows S
    ]
    for real, padded in bad:
        try:
            oracle.thd_meta(real, padded, S, lib=lib)
        except oracle.OracleValueError:
            continue
        raise AssertionError(f"no error for {real.tolist()} / {padded.tolist()}")


def pin_mask_standalone(lib):
    """_thd_padding_mask on a hand-checked layout, with and without padded
    lengths, and with a stream longer than the layout."""
    m = oracle.thd_padding_mask(12, np.array([3, 2, 6]), np.array([4, 2, 6]), lib=lib)
    assert m.tolist() == [False, False, False, True] + [False] * 8
    m = oracle.thd_padding_mask(9, np.array([3, 2]), None, lib=lib)
    assert m.tolist() == [False] * 5 + [True] * 4
    m = oracle.thd_padding_mask(10, np.array([1, 0, 2]), np.array([2, 3, 2]), lib=lib)
    assert m.tolist() == [False, True, True, True, True, False, False, True, True, True]


# --------------------------------------------------------------------------
# O5 trainer-side squeeze
# --------------------------------------------------------------------------
def pin_squeeze_page_example(lib):
    g = golden("who_packs_squeeze_example.json")
    src = np.asarray(g["rows"], np.int64)
    offs, mem = oracle.bins_to_csr(g["bins"])
    lens = np.asarray(g["input_lengths"], np.int64)
    t = g["trainer"]
    r = oracle.pack_squeeze(src, lens, offs, mem, g["multiple"], g["capacity"], t["stretch"], t["width"], lib=lib)
    assert r["packed"].shape == (1, t["width"])
    assert r["packed"].tolist() == t["packed"]
    assert r["cu_seqlens"][0].tolist() == t["cu_seqlens"]
    assert r["cu_seqlens_padded"][0].tolist() == t["cu_seqlens_padded"]
    assert r["max_total"] == t["width"]
    lo = g["loader"]
    r = oracle.pack_squeeze(src, lens, offs, mem, g["multiple"], g["capacity"], lo["stretch"], lo["width"], lib=lib)
    assert r["packed"].shape == (1, lo["width"])
    assert r["cu_seqlens"][0].tolist() == lo["cu_seqlens"]
    assert r["cu_seqlens_padded"][0].tolist() == lo["cu_seqlens_padded"]
    assert int((~r["padding_mask"]).sum()) == lo["real_tokens"]
    assert r["packed"][0, :t["width"]].tolist() == t["packed"][0]
    assert np.all(r["packed"][0, t["width"]:] == 0)


def pin_squeeze_closed_forms(lib, seeds=range(10)):
    """Real tokens of each bin, read in slot order, are the concatenation of
    its members' real prefixes; padded extents are multiples of m and start
    where the previous one ends; pad slots hold pad_value; mask marks them."""
    for seed in seeds:
        rng = np.random.default_rng(300 + seed)
        N, W = int(rng.integers(1, 9)), int(rng.integers(1, 12))
        m = int(rng.integers(1, 5))
        prob = synth.random_squeeze(rng, N, W, int(rng.integers(1, 4)))
        real, offs, mem = prob["real_lens"], prob["bin_offsets"], prob["bin_members"]
        need = max(sum(-(-int(real[i]) // m) * m for i in b) for b in prob["bins"])
        stretch = bool(seed % 2)
        cap = need + int(rng.integers(0, 5))
        width = cap if stretch else need + int(rng.integers(0, 3))
        r = oracle.pack_squeeze(prob["src"], real, offs, mem, m, cap, stretch, width, pad_value=-7, lib=lib)
        assert r["max_total"] == need
        for b, members in enumerate(prob["bins"]):
            row, mask = r["packed"][b], r["padding_mask"][b]
            want = np.concatenate([prob["src"][i, :real[i]] for i in members])
            assert np.array_equal(row[~mask], want)
            assert np.all(row[mask] == -7)
            cu, cup = r["cu_seqlens"][b], r["cu_seqlens_padded"][b]
            assert np.array_equal(np.diff(cu), real[members])
            widths = np.diff(cup)
            total = int(sum(-(-int(real[i]) // m) * m for i in members))
            if stretch:
                assert cup[-1] == cap
                assert np.all(widths[:-1] % m == 0)
            else:
                assert np.all(widths % m == 0) and cup[-1] == total
            for k, i in enumerate(members):
                assert not mask[cup[k]:cup[k] + real[i]].any()
                assert mask[cup[k] + real[i]:cup[k] + -(-int(real[i]) // m) * m].all()
            assert mask[total:].all()


def pin_squeeze_errors(lib):
    src = np.zeros((2, 8), np.int64)
    offs, mem = oracle.bins_to_csr([[0, 1]])
    try:
        oracle.pack_squeeze(src, np.array([5, 8]), offs, mem, 4, 12, False, 16, lib=lib)
        raise AssertionError("capacity overflow not reported")
    except oracle.OracleCapacityError:
        pass
    try:
        oracle.pack_squeeze(src, np.array([5, 8]), offs, mem, 4, 16, False, 12, lib=lib)
        raise AssertionError("width overflow not reported")
    except oracle.OracleCapacityError:
        pass
    # malformed input is reported ahead of a capacity problem in an earlier bin
    offs, mem = oracle.bins_to_csr([[0], [1, 5]])
    try:
        oracle.pack_squeeze(np.zeros((3, 8), np.int64), np.array([8, 1, 1]), offs, mem, 4, 4, False, 16, lib=lib)
        raise AssertionError("malformed bin not reported")
    except oracle.OracleValueError:
        pass
    for lens, bins in ((np.array([9, 1]), [[0, 1]]), (np.array([-1, 1]), [[0, 1]]),
                       (np.array([1, 1]), [[0], []]), (np.array([1, 1]), [[0, 2]])):
        offs, mem = oracle.bins_to_csr(bins)
        try:
            oracle.pack_squeeze(src, lens, offs, mem, 4, 64, False, 64, lib=lib)
        except oracle.OracleValueError:
            continue
        raise AssertionError(f"no error for {lens.tolist()} {bins}")


ALL_PINS = [
    pin_doc_ids_page_example,
    pin_doc_ids_brute_force,
    pin_doc_ids_invariants,
    pin_doc_ids_empty,
    pin_thd_page_example,
    pin_thd_closed_forms,
    pin_thd_full_rows_is_reshape,
    pin_thd_absorption,
    pin_thd_empty_and_filler_only,
    pin_thd_errors,
    pin_mask_standalone,
    pin_squeeze_page_example,
    pin_squeeze_closed_forms,
    pin_squeeze_errors,
]


# --------------------------------------------------------------------------
# O6 thd_padding_mask_from_token_ids
# --------------------------------------------------------------------------
def pin_mask_from_ids(lib):
    """Hand cases from the page's rule, then brute force: accepted exactly
    when the pad positions form a suffix (the mask never falls from True to
    False), and then the mask is the value comparison."""
    assert oracle.mask_from_token_ids(np.array([5, 6, 0, 0]), 0, lib=lib).tolist() == [False, False, True, True]
    assert oracle.mask_from_token_ids(np.array([5, 6, 7]), 0, lib=lib).tolist() == [False] * 3
    assert oracle.mask_from_token_ids(np.array([0, 0]), 0, lib=lib).tolist() == [True, True]
    assert oracle.mask_from_token_ids(np.zeros(0, np.int64), 0, lib=lib).tolist() == []
    for bad in ([5, 0, 6, 0], [0, 1], [3, 9, 9], [3, 3, 1, 3]):
        pad = 0 if 0 in bad else 3
        try:
            oracle.mask_from_token_ids(np.array(bad), pad, lib=lib)
        except oracle.OracleValueError:
            continue
        raise AssertionError(f"pad id inside content accepted: {bad}")
    for n in range(0, 8):
        for vals in itertools.product((0, 1, 2), repeat=n):
            ids = np.asarray(vals, np.int64)
            m = ids == 1
            ok = bool(np.all(np.diff(m.astype(int)) >= 0)) if n > 1 else True
            try:
                got = oracle.mask_from_token_ids(ids, 1, lib=lib)
                assert ok, (vals, "accepted")
                assert np.array_equal(got, m)
            except oracle.OracleValueError:
                assert not ok, (vals, "rejected")


# --------------------------------------------------------------------------
# O7 first-fit-decreasing
# --------------------------------------------------------------------------
def _bins_of(offs, mem):
    return [mem[offs[b]:offs[b + 1]].tolist() for b in range(len(offs) - 1)]


def _optimal_bins(sizes, capacity):
    """Brute force: fewest bins over every assignment (tiny inputs only)."""
    n = len(sizes)
    best = n
    for assign in itertools.product(range(n), repeat=n):
        if max(assign, default=-1) + 1 >= best:
            continue
        loads = [0] * n
        for i, b in enumerate(assign):
            loads[b] += sizes[i]
        if all(x <= capacity for x in loads):
            best = max(assign, default=-1) + 1
    return best


def pin_ffd(lib):
    offs, mem = oracle.ffd(np.array([4, 8, 1, 4, 2, 1]), 10, lib=lib)
    assert _bins_of(offs, mem) == [[1, 4], [0, 3, 2, 5]]
    g = golden("ffd_johnson_worst_case.json")
    offs, mem = oracle.ffd(np.array(g["sizes"]), g["capacity"], lib=lib)
    assert len(offs) - 1 == g["ffd_bins"]
    assert oracle.ffd(np.array([7, 7, 7]), 7, lib=lib)[0].size - 1 == 3
    assert oracle.ffd(np.array([1, 2, 3]), 100, lib=lib)[1].tolist() == [2, 1, 0]
    assert oracle.ffd(np.zeros(0, np.int64), 5, lib=lib)[0].tolist() == [0]
    try:
        oracle.ffd(np.array([3, 11]), 10, lib=lib)
        raise AssertionError("oversized item accepted")
    except oracle.OracleCapacityError:
        pass
    rng = np.random.default_rng(77)
    for trial in range(40):
        n = int(rng.integers(1, 7))
        cap = int(rng.integers(4, 12))
        sizes = rng.integers(1, cap + 1, size=n)
        offs, mem = oracle.ffd(sizes, cap, lib=lib)
        bins = _bins_of(offs, mem)
        assert sorted(mem.tolist()) == list(range(n))
        assert all(sum(sizes[i] for i in b) <= cap for b in bins)
        opt = _optimal_bins(list(sizes), cap)
        assert 9 * len(bins) <= 11 * opt + 6, (sizes, cap, bins, opt)  # FFD <= 11/9 OPT + 6/9
        # within a bin, items appear largest first (the visiting order)
        for b in bins:
            assert all((sizes[b[k]], -b[k]) >= (sizes[b[k + 1]], -b[k + 1]) for k in range(len(b) - 1))


# --------------------------------------------------------------------------
# O8 doc_ids -> pack lengths
# --------------------------------------------------------------------------
def pin_doc_ids_to_lengths(lib):
    r = oracle.doc_ids_to_lengths(np.array([[1, 1, 2, 2, 2, 0], [0, 0, 3, 3, 0, 4]], np.int32), 4, lib=lib)
    assert r["seq_lens"].tolist() == [[2, 3, -1000, -1000], [0, 2, 1, -1000]]
    assert r["seq_lens_padded"].tolist() == [[2, 4, -1000, -1000], [2, 3, 1, -1000]]
    assert r["position_ids"].tolist() == [[0, 1, 0, 1, 2, 0], [0, 0, 0, 1, 0, 0]]
    try:
        oracle.doc_ids_to_lengths(np.array([[1, 2, 3]], np.int32), 2, lib=lib)
        raise AssertionError("row over num_packs accepted")
    except oracle.OracleCapacityError:
        pass
    # random maps: padded lengths tile each row; real lengths are the
    # document runs (run-length encoding); the THD stream of the result is
    # the row-major flattening; sequence starts are segment starts of O1
    for seed in range(8):
        rng = np.random.default_rng(900 + seed)
        B, S = int(rng.integers(1, 4)), int(rng.integers(1, 30))
        d = synth.random_doc_ids(rng, B, S, "runs", np.int32)
        r = oracle.doc_ids_to_lengths(d, S, lib=lib)
        real, padded = r["seq_lens"], r["seq_lens_padded"]
        for b in range(B):
            keep = real[b] != -1000
            assert int(padded[b][keep].sum()) == S
            key = torch.from_numpy(d[b].astype(np.int64))
            vals, counts = torch.unique_consecutive(key, return_counts=True)
            doc_runs = [int(c) for v, c in zip(vals.tolist(), counts.tolist()) if v != 0]
            got = [int(x) for x in real[b][keep] if x > 0] if keep.any() else []
            assert got == doc_runs, (d[b].tolist(), real[b].tolist())
            for s in range(S):
                if d[b, s] == 0:
                    assert r["position_ids"][b, s] == 0
                else:
                    k = s
                    while k > 0 and d[b, k - 1] == d[b, s]:
                        k -= 1
                    assert r["position_ids"][b, s] == s - k
        out = oracle.process_input_for_thd({"input_ids": d.astype(np.int64), "seq_lens": real,
                                            "seq_lens_padded": padded}, lib=lib)
        assert np.array_equal(out["input_ids"], d.reshape(-1).astype(np.int64))
        seg_cu, _ = oracle.from_doc_ids(d, lib=lib)
        assert set(out["cu_seqlens_padded"][:-1].tolist()) <= set(seg_cu.tolist())


# --------------------------------------------------------------------------
# O9 split_batch_into_thd_chunks
# --------------------------------------------------------------------------
def pin_split_chunks(lib):
    g = golden("thd_utils_split_example.json")
    batch = {k: np.asarray(v, np.int64) for k, v in g["batch"].items()}
    r = oracle.split_batch_into_thd_chunks(batch, g["num_chunks"], lib=lib)
    assert r["input_ids"].tolist() == g["expected"]["input_ids"]
    assert r["cu_seqlens"].tolist() == g["expected"]["cu_seqlens"]
    assert r["labels"].shape == (2, 12) and r["padding_mask"].shape == (2, 12)
    one = oracle.split_batch_into_thd_chunks(batch, 1, lib=lib)
    assert one["cu_seqlens"].tolist() == [0, 6, 12, 18, 24]
    # ragged chunk tables are padded with the filler value
    batch2 = dict(batch)
    batch2["seq_lens"] = np.array([[3, 3], [6, -1000], [2, 4], [1, 5]])
    batch2["seq_lens_padded"] = np.array([[3, 3], [6, -1000], [2, 4], [1, 5]])
    r2 = oracle.split_batch_into_thd_chunks(batch2, 2, lib=lib)
    assert r2["cu_seqlens"].tolist() == [[0, 3, 6, 12, -1000], [0, 2, 6, 7, 12]]
    assert r2["num_sequences"].tolist() == [3, 4]
    for c in range(2):
        sub = {k: (v[c * 2:(c + 1) * 2]) for k, v in batch2.items()}
        single = oracle.process_input_for_thd(sub, lib=lib)
        assert np.array_equal(r2["input_ids"][c], single["input_ids"])
        assert r2["max_seqlen"][c] == single["max_seqlen"]
    # chunks with different stream lengths cannot be stacked
    batch3 = dict(batch2)
    batch3["seq_lens"] = np.array([[3, 3], [5, -1000], [2, 4], [1, 5]])
    batch3["seq_lens_padded"] = np.array([[3, 3], [5, -1000], [2, 4], [1, 5]])
    try:
        oracle.split_batch_into_thd_chunks(batch3, 2, lib=lib)
        raise AssertionError("unequal chunk streams stacked")
    except oracle.OracleValueError:
        pass
    try:
        oracle.split_batch_into_thd_chunks(batch, 3, lib=lib)
        raise AssertionError("num_chunks not dividing the batch accepted")
    except ValueError:
        pass


ALL_PINS += [pin_mask_from_ids, pin_ffd, pin_doc_ids_to_lengths, pin_split_chunks]

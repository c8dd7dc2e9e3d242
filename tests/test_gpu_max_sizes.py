"""Calls at the largest sizes the C ABI accepts, checked where the oracle can
follow (sampled rows) and by properties that hold at any size.

The inputs are built on the device (a few GB each); the oracle runs on the
sampled rows only.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

DEV = torch.device("cuda", 0)
INT32_MAX = 2**31 - 1


@pytest.fixture(scope="module", autouse=True)
def built():
    from varlen_attention_metadata_gb300 import build

    build.build()
    yield
    torch.cuda.empty_cache()


def info_of(t):
    return t[:16].view(torch.int32).tolist()[:4] if t.dtype == torch.uint8 else t[:4].tolist()


def test_doc_ids_scan_at_two_billion_tokens():
    import varlen_attention_metadata_gb300 as v

    B, S = 32768, 65535  # B*S = 2^31 - 2^15: 131070 tiles, far more than one wave
    N = B * S
    assert N <= INT32_MAX
    g = torch.Generator(device=DEV).manual_seed(5)
    # runs of about 64 tokens: a new document wherever a 1-in-64 draw hits
    starts = torch.randint(0, 64, (B, S), device=DEV, dtype=torch.int32, generator=g) == 0
    d = starts.to(torch.int32).cumsum(1, dtype=torch.int32)
    del starts
    cu, info = v.pseq_from_doc_ids(d)
    st, count, mx, total = info_of(info)
    assert st == 0 and total == N
    c = cu[: count + 1]
    assert int(c[0]) == 0 and int(c[-1]) == N
    assert bool((c[1:] > c[:-1]).all())
    # every row start is a boundary; boundaries per row equal the run count of the row
    row_first = torch.arange(B, device=DEV, dtype=torch.int64) * S
    pos = torch.searchsorted(c.to(torch.int64), row_first)
    assert bool((c.to(torch.int64)[pos] == row_first).all())
    assert mx == int((c[1:] - c[:-1]).max())
    # sampled rows against the oracle
    rng = np.random.default_rng(0)
    for b in sorted(rng.choice(B, size=16, replace=False).tolist()) + [0, B - 1]:
        row = d[b:b + 1].cpu().numpy()
        ref_cu, _ = oracle.from_doc_ids(row)
        lo = int(pos[b])
        hi = int(pos[b + 1]) if b + 1 < B else count
        got = c[lo:hi + 1].to(torch.int64).cpu().numpy() - b * S
        np.testing.assert_array_equal(got, ref_cu)
    del d, cu, c


@pytest.mark.parametrize("B,S", [(2, 2**30 - 1), (3, 715_827_882)])
def test_doc_ids_rows_at_the_widest(B, S):
    """One document per row at the widest rows a map can have (B*S just
    under 2^31): the boundaries are the row starts b*S, which the kernel
    finds with a precomputed reciprocal of S."""
    import varlen_attention_metadata_gb300 as v

    assert B * S <= INT32_MAX
    d = torch.full((B, S), 3, dtype=torch.int32, device=DEV)
    cu, info = v.pseq_from_doc_ids(d)
    assert info_of(info) == [0, B, S, B * S]
    assert cu[: B + 1].tolist() == [b * S for b in range(B + 1)]
    del d, cu


def test_squeeze_with_the_most_bins():
    import varlen_attention_metadata_gb300 as v

    nb = 65535  # the grid's second dimension
    rng = np.random.default_rng(6)
    W = 64
    real = rng.integers(0, W + 1, size=nb).astype(np.int64)
    src = rng.integers(-1000, 1000, size=(nb, W)).astype(np.int64)
    offs = np.arange(nb + 1, dtype=np.int32)
    mem = rng.permutation(nb).astype(np.int32)
    width = 64
    r = v.pack_squeeze(torch.from_numpy(src).to(DEV), torch.from_numpy(real).to(DEV),
                       (torch.from_numpy(offs).to(DEV), torch.from_numpy(mem).to(DEV)), 8, width, True, width, 7)
    st, count, mx, total = info_of(r["info"])
    ref = oracle.pack_squeeze(src, real, offs, mem, 8, width, True, width, 7)
    assert st == 0 and count == nb and total == ref["max_total"]
    np.testing.assert_array_equal(r["packed"].cpu().numpy(), ref["packed"])
    np.testing.assert_array_equal(r["padding_mask"].cpu().numpy(), ref["padding_mask"])
    np.testing.assert_array_equal(r["cu_seqlens"][: 2 * nb].cpu().numpy(), ref["cu_flat"])
    np.testing.assert_array_equal(r["cu_seqlens_padded"][: 2 * nb].cpu().numpy(), ref["cu_padded_flat"])
    # one bin more than the grid holds is refused before anything is enqueued
    offs2 = np.arange(nb + 2, dtype=np.int32)
    mem2 = np.arange(nb + 1, dtype=np.int32)
    real2 = np.ones(nb + 1, np.int64)
    src2 = np.zeros((nb + 1, 1), np.int64)
    with pytest.raises(Exception):
        v.pack_squeeze(torch.from_numpy(src2).to(DEV), torch.from_numpy(real2).to(DEV),
                       (torch.from_numpy(offs2).to(DEV), torch.from_numpy(mem2).to(DEV)), 1, 1, False, 1, 0)


def test_token_mask_at_the_int32_limit():
    import varlen_attention_metadata_gb300 as v

    n = INT32_MAX
    tail = 1 << 20
    g = torch.Generator(device=DEV).manual_seed(7)
    ids = torch.randint(1, 32000, (n,), device=DEV, dtype=torch.int32, generator=g)
    ids[n - tail:] = 0
    mask, info = v.thd_mask_from_token_ids(ids, 0)
    st, count, _, total = info_of(info)
    assert st == 0 and count == tail and total == n
    assert int(mask[: n - tail].sum(dtype=torch.int64)) == 0 and bool(mask[n - tail:].all())
    # a pad id inside the content is refused
    ids[12345] = 0
    _, info = v.thd_mask_from_token_ids(ids, 0)
    assert info_of(info)[0] == 3
    # sampled windows against the oracle
    ids[12345] = 7
    rng = np.random.default_rng(1)
    for start in [0, n - tail - 100, n - 4096] + rng.integers(0, n - tail - 4096, size=6).tolist():
        win = ids[start:start + 4096].cpu().numpy()  # content, then possibly the pad tail: a valid stream
        got = mask[start:start + 4096].cpu().numpy().astype(bool)
        np.testing.assert_array_equal(got, oracle.mask_from_token_ids(win, 0))
    del ids, mask


def test_thd_conversion_at_two_billion_tokens():
    import varlen_attention_metadata_gb300 as v

    B, S, P = 32768, 65535, 8  # 2^31 - 2^15 source slots, 262144 table entries: the two-kernel path
    rng = np.random.default_rng(8)
    real = np.full((B, P), -1000, np.int64)
    padded = np.full((B, P), -1000, np.int64)
    for b in range(B):
        k = int(rng.integers(1, P + 1))
        used = int(rng.integers(k, S + 1))  # rows may end short of S
        cuts = np.sort(rng.choice(np.arange(1, used), size=k - 1, replace=False)) if k > 1 else np.array([], int)
        pl = np.diff(np.concatenate([[0], cuts, [used]]))
        rl = pl - rng.integers(0, np.minimum(pl, 4))
        slots = np.sort(rng.choice(P, size=k, replace=False))  # filler between kept entries too
        padded[b, slots] = pl
        real[b, slots] = rl
    g = torch.Generator(device=DEV).manual_seed(9)
    ids = torch.randint(-2**31, 2**31 - 1, (B, S), device=DEV, dtype=torch.int32, generator=g)
    r = v.thd_from_batch(torch.from_numpy(real).to(DEV), torch.from_numpy(padded).to(DEV), S, [(ids, 1)])
    st, n, mx, T = info_of(r["info"])
    meta = oracle.thd_meta(real, padded, S)
    assert st == 0 and n == meta["num_sequences"] and T == meta["total_tokens"] and mx == meta["max_seqlen"]
    np.testing.assert_array_equal(r["cu_seqlens"][: n + 1].cpu().numpy(), meta["cu_seqlens"])
    np.testing.assert_array_equal(r["cu_seqlens_padded"][: n + 1].cpu().numpy(), meta["cu_seqlens_padded"])
    mask = r["padding_mask"][:T]
    assert int(mask.sum(dtype=torch.int64)) == T - int(meta["seq_real"].sum())
    out = r["dst"][0][0]
    # sampled rows: the row's stream slice against the oracle on that row alone
    first_seq = np.concatenate([[0], np.cumsum((real != -1000).sum(axis=1))])
    cup = meta["cu_seqlens_padded"]
    for b in sorted(rng.choice(B, size=12, replace=False).tolist()) + [0, B - 1]:
        ref = oracle.process_input_for_thd({"input_ids": ids[b:b + 1].cpu().numpy(), "seq_lens": real[b:b + 1],
                                            "seq_lens_padded": padded[b:b + 1]}, absorb=False)
        lo, hi = int(cup[first_seq[b]]), int(cup[first_seq[b + 1]])
        np.testing.assert_array_equal(out[lo:hi].cpu().numpy(), ref["input_ids"])
        np.testing.assert_array_equal(mask[lo:hi].cpu().numpy(), ref["padding_mask"])
    del ids, r, out, mask


def test_bridge_with_the_most_rows():
    import varlen_attention_metadata_gb300 as v

    B, S, P = 65535, 32768, 1024  # 65535 rows is the grid's limit; B*S = 2^31 - 2^15
    g = torch.Generator(device=DEV).manual_seed(10)
    draw = torch.randint(0, 64, (B, S), device=DEV, dtype=torch.int32, generator=g)
    # documents of about 64 tokens, a padding run wherever a 1-in-16 draw hits a run start
    starts = draw == 0
    d = starts.to(torch.int32).cumsum(1, dtype=torch.int32)
    d = torch.where((d % 16) == 5, torch.zeros_like(d), d)
    del draw, starts
    real, padded, pos, info = v.pseq_doc_ids_to_lengths(d, P)
    st, most, longest, total = info_of(info)
    assert st == 0
    kept = real != -1000
    assert total == int(kept.sum()) and most == int(kept.sum(dim=1).max())
    # padded lengths tile every row
    assert bool((torch.where(kept, padded, torch.zeros_like(padded)).sum(dim=1) == S).all())
    rng = np.random.default_rng(2)
    for b in sorted(rng.choice(B, size=12, replace=False).tolist()) + [0, B - 1]:
        ref = oracle.doc_ids_to_lengths(d[b:b + 1].cpu().numpy(), P)
        np.testing.assert_array_equal(real[b:b + 1].cpu().numpy(), ref["seq_lens"])
        np.testing.assert_array_equal(padded[b:b + 1].cpu().numpy(), ref["seq_lens_padded"])
        np.testing.assert_array_equal(pos[b:b + 1].cpu().numpy(), ref["position_ids"])
    del d, real, padded, pos

"""CUDA path against the CPU oracle for split_batch_into_thd_chunks,
thd_padding_mask_from_token_ids, first-fit-decreasing and the doc_ids ->
pack-lengths bridge (bit-exact; every call through the C ABI)."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from varlen_attention_metadata_gb300 import build

    build.build()
    yield


def V():
    import varlen_attention_metadata_gb300 as v

    return v


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def info_of(block):
    return tuple(block[:16].view(torch.int32).tolist())


def golden(name):
    with open(os.path.join(os.path.dirname(__file__), "golden", name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------
# thd_padding_mask_from_token_ids
# --------------------------------------------------------------------------
def check_token_mask(ids: np.ndarray, pad: int, offset: int = 0):
    v = V()
    flat = torch.zeros(ids.size + offset, dtype=torch.int32 if ids.dtype == np.int32 else torch.int64, device=DEV)
    x = flat[offset:]
    x.copy_(torch.from_numpy(ids))
    mask, info = v.thd_mask_from_token_ids(x, pad)
    st, count, _, total = info_of(info)
    try:
        ref = oracle.mask_from_token_ids(ids, pad)
    except oracle.OracleValueError:
        assert st == 3
        return
    assert st == 0 and total == ids.size and count == int(ref.sum())
    np.testing.assert_array_equal(mask.cpu().numpy(), ref)


@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_token_mask_random(dtype):
    rng = np.random.default_rng(3)
    for n in (0, 1, 7, 8, 9, 1000, 4097, 65536 + 13, 3_000_001):
        content = rng.integers(1, 32000, size=n).astype(dtype)
        tail = int(rng.integers(0, n + 1)) if n else 0
        good = content.copy()
        if tail:
            good[n - tail:] = 0
        check_token_mask(good, 0)
        check_token_mask(good, 0, offset=1)  # unaligned: scalar path
        if n > 2:
            bad = good.copy()
            bad[int(rng.integers(0, max(1, n - tail - 1)))] = 0  # pad id inside the content
            check_token_mask(bad, 0)
        check_token_mask(content, 7)  # a pad id that may not occur at all


def test_token_mask_extreme_values():
    # a pad id that shares its low 32 bits with content ids, and negative
    # or limit pad ids: the comparison is on the whole value
    rng = np.random.default_rng(21)
    cases = [(np.int64, 1 << 32, np.array([0, 1 << 33, (1 << 32) + 1, -1, np.iinfo(np.int64).min], np.int64)),
             (np.int64, -1, np.array([np.iinfo(np.int64).max, 1, 0, (1 << 32) - 1], np.int64)),
             (np.int32, np.iinfo(np.int32).min, np.array([0, 1, -1, np.iinfo(np.int32).max], np.int32))]
    for dtype, pad, content_pool in cases:
        for n in (9, 4096 + 3, 100_001):
            ids = content_pool[rng.integers(0, len(content_pool), size=n)].astype(dtype)
            tail = int(rng.integers(0, n + 1))
            if tail:
                ids[n - tail:] = pad
            check_token_mask(ids, pad)
            check_token_mask(ids, pad, offset=1)
            if tail > 1 and n - tail > 1:
                bad = ids.copy()
                bad[int(rng.integers(0, n - tail))] = pad  # the pad id inside the content
                check_token_mask(bad, pad)


def test_token_mask_page_rule_and_api():
    v = V()
    m = v.thd_padding_mask_from_token_ids(dev(np.array([5, 6, 0, 0])), 0)
    assert m.tolist() == [False, False, True, True]
    with pytest.raises(ValueError):
        v.thd_padding_mask_from_token_ids(dev(np.array([5, 0, 6, 0])), 0)
    # workspace reuse across calls of different sizes
    rng = np.random.default_rng(9)
    for n in (100_000, 17, 2_000_000, 5):
        ids = rng.integers(1, 9, size=n).astype(np.int64)
        ids[n // 2:] = 0
        check_token_mask(ids, 0)


# --------------------------------------------------------------------------
# first-fit-decreasing
# --------------------------------------------------------------------------
def check_ffd(lens: np.ndarray, capacity: int, multiple: int = 1):
    v = V()
    offs, mem, info = v.pack_ffd(dev(lens.astype(np.int64)), capacity, multiple)
    st, nb, fullest, total = info_of(info)
    sizes = -(-lens.astype(np.int64) // multiple) * multiple
    try:
        ref_offs, ref_mem = oracle.ffd(sizes if (lens >= 0).all() else lens, capacity)
    except oracle.OracleCapacityError:
        assert st == 4
        return None
    except oracle.OracleValueError:
        assert st == 3
        return None
    assert st == 0 and nb == len(ref_offs) - 1
    np.testing.assert_array_equal(offs[: nb + 1].cpu().numpy(), ref_offs)
    np.testing.assert_array_equal(mem.cpu().numpy(), ref_mem)
    assert total == int(sizes.sum())
    loads = [int(sizes[ref_mem[ref_offs[b]:ref_offs[b + 1]]].sum()) for b in range(nb)]
    assert fullest == (max(loads) if loads else 0)
    return ref_offs, ref_mem


def test_ffd_examples():
    check_ffd(np.array([4, 8, 1, 4, 2, 1]), 10)
    g = golden("ffd_johnson_worst_case.json")
    offs, _ = check_ffd(np.array(g["sizes"]), g["capacity"])
    assert len(offs) - 1 == g["ffd_bins"]
    check_ffd(np.zeros(0, np.int64), 10)
    check_ffd(np.array([5, 11, 2]), 10)   # an item over capacity
    check_ffd(np.array([5, -1, 2]), 10)   # a negative length


@pytest.mark.parametrize("n", [1, 2, 17, 31, 32, 33, 64, 256, 1000, 1024, 1025, 4097, 8192])
def test_ffd_random(n):
    rng = np.random.default_rng(n)
    for multiple in (1, 64):
        lens = np.clip(np.round(rng.lognormal(6.5, 0.8, size=n)), 1, 4096).astype(np.int64)
        check_ffd(lens, 32768, multiple)
        check_ffd(rng.integers(1, 50, size=n), int(rng.integers(50, 400)), multiple)


def test_ffd_equal_size_runs():
    # runs of equal sizes: zero sizes, runs longer than a warp, a run that
    # opens the 33rd bin half way, runs that first top up open bins and then
    # open new ones
    check_ffd(np.zeros(50, np.int64), 10)
    check_ffd(np.array([0] * 5 + [3] * 40 + [0] * 7), 10)
    check_ffd(np.array([6] * 40), 10)
    check_ffd(np.array([5] * 100), 10)
    check_ffd(np.array([7] * 3 + [3] * 50), 10)
    check_ffd(np.array([9] * 31 + [1] * 70 + [4] * 9), 10)
    check_ffd(np.arange(1, 65), 4096, 64)  # every size rounds to 64
    rng = np.random.default_rng(5)
    for n in (300, 5000):
        check_ffd(rng.choice([0, 1, 2, 3, 5, 8], size=n), 17)
        check_ffd(rng.choice([16, 48, 64, 100], size=n), 128)


def test_ffd_feeds_the_squeeze():
    """The squeeze workload, with bins from the GPU packer."""
    v = V()
    c = synth.squeeze(0)
    offs, mem = v.first_fit_decreasing(dev(c["real_lens"]), c["capacity"], c["multiple"])
    np.testing.assert_array_equal(offs.cpu().numpy(), c["bin_offsets"])
    np.testing.assert_array_equal(mem.cpu().numpy(), c["bin_members"])
    r = v.squeeze_bins(dev(c["src"]), dev(c["real_lens"]), (offs, mem), c["multiple"], c["capacity"],
                       stretch_to_capacity=True)
    ref = oracle.pack_squeeze(c["src"], c["real_lens"], c["bin_offsets"], c["bin_members"], c["multiple"],
                              c["capacity"], True, c["capacity"])
    np.testing.assert_array_equal(r["packed_input_ids"].cpu().numpy(), ref["packed"])


# --------------------------------------------------------------------------
# doc_ids -> seq_lens bridge
# --------------------------------------------------------------------------
def check_bridge(d: np.ndarray, num_packs: int):
    v = V()
    real, padded, pos, info = v.pseq_doc_ids_to_lengths(dev(d), num_packs)
    st, most, longest, total = info_of(info)
    try:
        ref = oracle.doc_ids_to_lengths(d, num_packs)
    except oracle.OracleCapacityError:
        assert st == 4
        return
    assert st == 0
    np.testing.assert_array_equal(real.cpu().numpy(), ref["seq_lens"])
    np.testing.assert_array_equal(padded.cpu().numpy(), ref["seq_lens_padded"])
    np.testing.assert_array_equal(pos.cpu().numpy(), ref["position_ids"])
    kept = ref["seq_lens"] != -1000
    assert most == int(kept.sum(axis=1).max(initial=0)) and total == int(kept.sum())
    assert longest == int(ref["seq_lens"][kept].max(initial=0))


@pytest.mark.parametrize("kind", ["runs", "iid", "zeros", "const", "alternating", "long"])
def test_bridge_random(kind):
    rng = np.random.default_rng(31)
    for B, S in ((1, 1), (2, 7), (3, 4096), (2, 4097), (5, 9000), (1, 20000)):
        for dtype in (np.int32, np.int64):
            d = synth.random_doc_ids(rng, B, S, kind, dtype)
            check_bridge(d, S)
    d = synth.random_doc_ids(rng, 3, 500, "runs", np.int32)
    check_bridge(d, 4)  # rows hold more sequences than slots


@pytest.mark.parametrize("chunks", [1, 2, 9])
def test_bridge_chunk_boundaries(chunks):
    """Rows ending one token before, on and one token after a chunk boundary
    (4096 tokens a chunk), so the last chunk is full, nearly empty or one
    token long, and the row's fill CTA follows 1, 2 or 9 chunks."""
    rng = np.random.default_rng(41 + chunks)
    for S in (chunks * 4096 - 1, chunks * 4096, chunks * 4096 + 1):
        for kind in ("runs", "alternating"):
            check_bridge(synth.random_doc_ids(rng, 3, S, kind, np.int32), S)


def test_bridge_overflow_with_many_chunks():
    """Rows of several 4096-token chunks holding more sequences than slots:
    the walk writes only the slots that exist, the row's fill CTA has
    nothing to fill, and the call reports PSEQ_ERR_CAPACITY; with exactly as
    many slots as the fullest row needs it is exact."""
    rng = np.random.default_rng(37)
    for kind in ("runs", "iid", "alternating"):
        d = synth.random_doc_ids(rng, 3, 5 * 4096 + 77, kind, np.int32)
        check_bridge(d, 16)
        ref = oracle.doc_ids_to_lengths(d, d.shape[1])
        need = int((ref["seq_lens"] != -1000).sum(axis=1).max())
        check_bridge(d, need)


def test_bridge_extreme_values():
    # non-zero ids whose low 32 bits are zero are documents, not padding;
    # negative ids and the type's limits are documents too
    rng = np.random.default_rng(43)
    pool64 = np.array([0, 1, -1, 1 << 32, 1 << 33, (1 << 32) + 1, np.iinfo(np.int64).max,
                       np.iinfo(np.int64).min], np.int64)
    pool32 = np.array([0, 1, -1, 1 << 16, np.iinfo(np.int32).max, np.iinfo(np.int32).min], np.int32)
    for pool in (pool64, pool32):
        for B, S in ((3, 40), (2, 9000), (1, 40000)):
            flat = np.empty(B * S, pool.dtype)
            pos = 0
            while pos < B * S:
                L = int(rng.geometric(0.2))
                flat[pos:pos + L] = pool[rng.integers(0, len(pool))]
                pos += L
            check_bridge(flat.reshape(B, S), S)


def test_bridge_long_rows():
    # rows of 35 and 49 chunks: the look-back takes more than one round of 32
    rng = np.random.default_rng(41)
    for S, kind in ((140_001, "runs"), (200_000, "long"), (200_000, "runs")):
        d = synth.random_doc_ids(rng, 2, S, kind, np.int32)
        check_bridge(d, S)


def test_bridge_workloads():
    check_bridge(synth.doc_map_small(0)["doc_ids"], 64)
    check_bridge(synth.doc_map_stress(0), 8192)


def test_bridge_round_trip_through_thd():
    v = V()
    c = synth.doc_map_small(2)
    lens = v.doc_ids_to_seq_lens(dev(c["doc_ids"]))
    out = v.process_input_for_thd({"input_ids": dev(c["input_ids"]), "seq_lens": lens["seq_lens"],
                                   "seq_lens_padded": lens["seq_lens_padded"], "position_ids": lens["position_ids"]})
    np.testing.assert_array_equal(out["input_ids"].cpu().numpy(), c["input_ids"].reshape(-1))
    np.testing.assert_array_equal(out["position_ids"].cpu().numpy(), c["position_ids"].reshape(-1))


# --------------------------------------------------------------------------
# split_batch_into_thd_chunks
# --------------------------------------------------------------------------
def check_split(batch_np: dict, num_chunks: int, hidden=None, absorb=True):
    v = V()
    real, padded = batch_np["seq_lens"], batch_np.get("seq_lens_padded")
    ids = batch_np["input_ids"]
    B, S = ids.shape[:2]
    fields_np = [(ids, 1)]
    if "position_ids" in batch_np:
        pos = batch_np["position_ids"]
        fields_np.append((pos, pos.shape[0] if pos.ndim == 3 else 1))
    fields_t = [(dev(a), p) for a, p in fields_np] + ([(hidden, 1)] if hidden is not None else [])
    r = v.thd_chunks_from_batch(dev(real), None if padded is None else dev(padded), S, num_chunks, fields_t, -1000,
                                absorb)
    infos = r["infos"].cpu().numpy()
    Bc = B // num_chunks
    Sc = Bc * S  # chunk c's stream starts c * planes * Sc rows in, its mask c * Sc bytes in: defined for any lengths
    for c in range(num_chunks):
        sl = slice(c * Bc, (c + 1) * Bc)
        try:
            meta = oracle.thd_meta(real[sl], None if padded is None else padded[sl], S, -1000, absorb)
        except oracle.OracleValueError:
            assert infos[c, 0] == 3
            continue
        st, n, mx, T = infos[c]
        assert st == 0 and n == meta["num_sequences"] and T == meta["total_tokens"] and mx == meta["max_seqlen"]
        row = r["cu_seqlens"][c].cpu().numpy()
        np.testing.assert_array_equal(row[: n + 1], meta["cu_seqlens"])
        assert np.all(row[n + 1:] == -1000)
        if padded is not None:
            rowp = r["cu_seqlens_padded"][c].cpu().numpy()
            np.testing.assert_array_equal(rowp[: n + 1], meta["cu_seqlens_padded"])
            assert np.all(rowp[n + 1:] == -1000)
        assert bool(r["pad_between"][c].item()) == meta["pad_between_seqs"]
        for (a, planes), (dst, _, rowshape) in zip(fields_np, r["dst"]):
            sub = a[:, sl] if planes > 1 else a[sl]
            want = oracle.thd_gather(sub, meta, Bc, S, planes=planes)
            start = c * planes * Sc
            got = dst[start:start + want.size].cpu().numpy().reshape(want.shape)
            np.testing.assert_array_equal(got, want)
        if hidden is not None:
            h = hidden[sl].cpu().view(torch.int16).numpy()
            want = oracle.thd_gather(h, meta, Bc, S)
            row = h.shape[2]
            got = r["dst"][-1][0][c * Sc * row:c * Sc * row + want.size].cpu().view(torch.int16).numpy()
            np.testing.assert_array_equal(got.reshape(want.shape), want)
        m = r["padding_mask"][c * Sc:c * Sc + T].cpu().numpy()
        np.testing.assert_array_equal(m, oracle.thd_padding_mask(T, meta["seq_real"],
                                                                 meta["seq_padded"] if padded is not None else None))


def test_split_page_example():
    v = V()
    g = golden("thd_utils_split_example.json")
    batch = {k: np.asarray(x, np.int64) for k, x in g["batch"].items()}
    check_split(batch, g["num_chunks"])
    out = v.split_batch_into_thd_chunks({k: dev(x) for k, x in batch.items()}, g["num_chunks"])
    assert out["input_ids"].tolist() == g["expected"]["input_ids"]
    assert out["cu_seqlens"].tolist() == g["expected"]["cu_seqlens"]
    ref = oracle.split_batch_into_thd_chunks(batch, g["num_chunks"])
    for k in ("input_ids", "labels", "position_ids", "padding_mask", "cu_seqlens", "cu_seqlens_padded"):
        np.testing.assert_array_equal(out[k].cpu().numpy(), ref[k])
    np.testing.assert_array_equal(out["max_seqlen"].cpu().numpy(), ref["max_seqlen"])
    np.testing.assert_array_equal(out["pad_between_seqs"].cpu().numpy(), ref["pad_between_seqs"])


@pytest.mark.parametrize("seed", range(4))
def test_split_random(seed):
    rng = np.random.default_rng(40 + seed)
    B, S, P = 8, int(rng.integers(8, 600)), int(rng.integers(1, 12))
    real, padded = synth.random_thd(rng, B, S, P, multiple=4, fill_rows=bool(seed % 2))
    batch = {"input_ids": rng.integers(0, 32000, size=(B, S)).astype(np.int64),
             "position_ids": rng.integers(0, 99, size=(3, B, S)).astype(np.int64),
             "seq_lens": real, "seq_lens_padded": padded}
    hidden = torch.randn(B, S, 6, device=DEV).to(torch.bfloat16)
    for nc in (1, 2, 4, 8):
        check_split(batch, nc, hidden=hidden, absorb=bool(nc % 2))
    # the page-level function stacks or refuses
    v = V()
    tb = {k: dev(a) for k, a in batch.items()}
    for nc in (2, 4):
        try:
            ref = oracle.split_batch_into_thd_chunks(batch, nc)
        except oracle.OracleValueError:
            with pytest.raises(ValueError):
                v.split_batch_into_thd_chunks(tb, nc)
            continue
        out = v.split_batch_into_thd_chunks(tb, nc)
        for k in ("input_ids", "position_ids", "padding_mask", "cu_seqlens", "cu_seqlens_padded"):
            np.testing.assert_array_equal(out[k].cpu().numpy(), ref[k])


def test_split_large_chunk_tables():
    rng = np.random.default_rng(77)
    B, S, P = 4, 3000, 1200  # 2400 entries per chunk of 2 rows: two-kernel path
    real, padded = synth.random_thd(rng, B, S, P, multiple=1, fill_rows=True)
    batch = {"input_ids": rng.integers(0, 32000, size=(B, S)).astype(np.int64), "seq_lens": real,
             "seq_lens_padded": padded}
    check_split(batch, 2)


def test_split_unequal_chunks_rejected():
    v = V()
    batch = {"input_ids": dev(np.zeros((4, 6), np.int64)),
             "seq_lens": dev(np.array([[3, 3], [5, -1000], [2, 4], [1, 5]])),
             "seq_lens_padded": dev(np.array([[3, 3], [5, -1000], [2, 4], [1, 5]]))}
    with pytest.raises(ValueError):
        v.split_batch_into_thd_chunks(batch, 2)

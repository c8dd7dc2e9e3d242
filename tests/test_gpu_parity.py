"""CUDA path against the CPU oracle, element by element (tolerance 0: all of
this work is integer, index or bit-copy work).

Every call goes through the C ABI of libpseq.so (ctypes binding).  Sizes
span several tiles with ragged tails; the five workloads run at full size.
"""
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
    import varlen_attention_metadata_gb300 as v

    v.load_library()
    yield


def V():
    import varlen_attention_metadata_gb300 as v

    return v


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def info_of(block):
    return tuple(block[:16].view(torch.int32).tolist())


CANARY = 0x5A


# --------------------------------------------------------------------------
# pseq_from_doc_ids
# --------------------------------------------------------------------------
def run_doc_ids(d: np.ndarray, offset_elems: int = 0):
    """Run the scan; optionally place doc_ids at an element offset so the
    pointer is not 16-byte aligned.  Returns (cu, info, canary_ok)."""
    v = V()
    B, S = d.shape
    flat = torch.zeros(B * S + offset_elems, dtype=torch.int32 if d.dtype == np.int32 else torch.int64, device=DEV)
    src = flat[offset_elems:]
    src.copy_(torch.from_numpy(d.reshape(-1)))
    src = src.view(B, S)
    guard = 16
    cu_full = torch.full((B * S + 1 + 2 * guard,), CANARY, dtype=torch.int32, device=DEV)
    cu = cu_full[guard:guard + B * S + 1]
    _, info = v.pseq_from_doc_ids(src, cu_seqlens=cu)
    st, count, mx, total = info_of(info)
    host = cu_full.cpu().numpy()
    canary_ok = (np.all(host[:guard] == CANARY) and np.all(host[guard + count + 1:] == CANARY))
    return host[guard:guard + count + 1], (st, count, mx, total), canary_ok


def check_doc_ids(d, offset_elems=0):
    cu, (st, count, mx, total), canary_ok = run_doc_ids(d, offset_elems)
    ref_cu, ref_mx = oracle.from_doc_ids(d)
    assert st == 0
    assert canary_ok, "write outside cu_seqlens[0 .. num_segments]"
    assert count == len(ref_cu) - 1
    np.testing.assert_array_equal(cu, ref_cu)
    assert mx == ref_mx
    assert total == d.size


def test_doc_ids_page_example():
    check_doc_ids(np.array([[1, 1, 2, 2, 2, 0]], np.int32))


@pytest.mark.parametrize("kind", ["runs", "iid", "zeros", "const", "alternating", "long"])
@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_doc_ids_random(kind, dtype):
    rng = np.random.default_rng(7)
    shapes = [(1, 1), (1, 7), (3, 1), (2, 5), (5, 4096), (3, 4097), (7, 1500), (1, 3 * 16384 + 123),
              (13, 2049), (40, 1), (2, 16385)]
    for B, S in shapes:
        d = synth.random_doc_ids(rng, B, S, kind, dtype)
        check_doc_ids(d)
        check_doc_ids(d, offset_elems=1)  # unaligned pointer: scalar load path


def extreme_runs(rng, pool, B, S):
    """Runs of values drawn from `pool` (mean length 5)."""
    flat = np.empty(B * S, pool.dtype)
    pos = 0
    while pos < B * S:
        L = int(rng.geometric(0.2))
        flat[pos:pos + L] = pool[rng.integers(0, len(pool))]
        pos += L
    return flat.reshape(B, S)


INT64_POOL = np.array([0, 1, -1, 1 << 32, (1 << 32) + 1, 1 << 33, -(1 << 40), np.iinfo(np.int64).max,
                       np.iinfo(np.int64).min], np.int64)
INT32_POOL = np.array([0, 1, -1, 1 << 16, np.iinfo(np.int32).max, np.iinfo(np.int32).min], np.int32)


@pytest.mark.parametrize("dtype", [np.int32, np.int64])
def test_doc_ids_extreme_values(dtype):
    # ids that differ only in their high 32 bits, negative ids and the type's
    # limits: boundaries are decided on the whole value
    rng = np.random.default_rng(77)
    pool = INT64_POOL if dtype == np.int64 else INT32_POOL
    for B, S in ((3, 40), (2, 20000), (1, 70001)):
        d = extreme_runs(rng, pool, B, S)
        check_doc_ids(d)
        check_doc_ids(d, offset_elems=1)


def test_doc_ids_many_tiles_chain():
    """Over a hundred tiles, so the look-back crosses several 32-tile windows."""
    rng = np.random.default_rng(11)
    d = synth.random_doc_ids(rng, 9, 200_003, "runs", np.int32)
    check_doc_ids(d)
    d = synth.random_doc_ids(rng, 2, 700_001, "long", np.int32)  # tiles with no boundary at all
    check_doc_ids(d)


def test_doc_ids_long_lookback():
    """Over 500 tiles: long look-back chains."""
    rng = np.random.default_rng(12)
    check_doc_ids(synth.random_doc_ids(rng, 4, 2_200_001, "runs", np.int32))


@pytest.mark.parametrize("tiles", [1, 2, 128, 129, 130])
def test_doc_ids_tile_and_round_boundaries(tiles):
    """Maps that end exactly on a tile, one token short of one and one token
    into the next; 128 to 130 tiles put the last tiles at the edge of one
    look-back round (128 predecessors per round)."""
    rng = np.random.default_rng(tiles)
    for n in (tiles * 16384 - 1, tiles * 16384, tiles * 16384 + 1):
        B = 2 if n % 2 == 0 else 1
        check_doc_ids(synth.random_doc_ids(rng, B, n // B, "runs", np.int32))


def test_doc_ids_empty():
    v = V()
    for shape in ((0, 5), (4, 0)):
        d = torch.zeros(shape, dtype=torch.int32, device=DEV)
        p = v.packed_seq_params_from_doc_ids(d)
        assert p.cu_seqlens.tolist() == [0] and p.max_seqlen == 0


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_doc_ids_small_map_workload(seed):
    check_doc_ids(synth.doc_map_small(seed)["doc_ids"])


@pytest.mark.parametrize("seed", [0, 1])
def test_doc_ids_stress_map_workload(seed):
    check_doc_ids(synth.doc_map_stress(seed))


def test_doc_ids_workspace_serves_any_sequence_of_calls():
    """Back-to-back calls of different sizes on one cached workspace: slots
    of an earlier, bigger map are never read as this call's."""
    rng = np.random.default_rng(3)
    for S in (50_000, 4096 * 5, 999, 120_000, 7):
        check_doc_ids(synth.random_doc_ids(rng, 3, S, "runs", np.int32))


def row_start_widths():
    widths = set(range(1, 40))
    for k in range(5, 27):
        widths |= {2**k - 1, 2**k, 2**k + 1}
    return sorted(widths | {3 * 16384 + 5, 65535, 100_003, 1_000_003})


@pytest.mark.parametrize("dtype", [torch.int32, torch.int64])
def test_doc_ids_row_starts_at_every_width(dtype):
    """One document filling every row: the boundaries are exactly the row
    starts b*S, whatever the row width (the kernel finds them with a
    precomputed reciprocal of S instead of a division).  At least three rows,
    so the quotients reach 2; up to 2^26 tokens."""
    v = V()
    for S in row_start_widths():
        B = max(3, min(4096, (1 << 26) // S))
        x = torch.full((B, S), 5, dtype=dtype, device=DEV)
        cu, info = v.pseq_from_doc_ids(x)
        assert info_of(info) == (0, B, S, B * S), S
        assert torch.equal(cu[: B + 1].to(torch.int64), torch.arange(0, B * S + 1, S, device=DEV)), S
        del x, cu


def test_doc_ids_random_at_widths_near_powers_of_two():
    rng = np.random.default_rng(17)
    for S in (15, 16, 17, 31, 33, 255, 257, 1023, 1025, 16383, 16384, 16385, 32767, 32769):
        B = max(2, 120_000 // S)
        check_doc_ids(synth.random_doc_ids(rng, B, S, "runs", np.int32))


def raw_scan(d: np.ndarray, ws: torch.Tensor):
    """pseq_from_doc_ids through the C ABI with the caller's workspace."""
    import ctypes

    v = V()
    lib = v.load_library()
    B, S = d.shape
    x = dev(d)
    cu = torch.empty(B * S + 1, dtype=torch.int32, device=DEV)
    info = torch.zeros(32, dtype=torch.uint8, device=DEV)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.pseq_from_doc_ids(P(x), x.element_size(), B, S, P(cu), P(info), P(ws), ws.numel(),
                               ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0
    return cu, info_of(info)


def header_tag(ws: torch.Tensor) -> int:
    """The workspace header's first word: the last call's tag (little-endian)."""
    return int(ws[:8].cpu().numpy().view(np.uint64)[0])


def check_raw(d, ws):
    cu, (st, count, mx, total) = raw_scan(d, ws)
    ref_cu, ref_mx = oracle.from_doc_ids(d)
    assert (st, count, mx, total) == (0, len(ref_cu) - 1, ref_mx, d.size)
    np.testing.assert_array_equal(cu[:count + 1].cpu().numpy(), ref_cu)


@pytest.mark.parametrize("withheld", [None, 1])
def test_doc_ids_tag_wraps_around(withheld):
    """Each call stamps its slots with the header's tag plus one.  The call
    that takes the last tag (2^32 - 1) zero-fills the whole buffer, slots of
    earlier bigger maps included, and resets the header, also when one of
    its tiles failed; the calls around it are exact."""
    v = V()
    lib = v.load_library()
    rng = np.random.default_rng(21)
    big = synth.random_doc_ids(rng, 6, 80_000, "runs", np.int32)    # 30 tiles
    small = synth.random_doc_ids(rng, 3, 50_000, "runs", np.int32)  # 10 tiles
    ws = torch.zeros(lib.pseq_from_doc_ids_workspace_size(*big.shape) + 1000, dtype=torch.uint8, device=DEV)
    check_raw(big, ws)
    assert header_tag(ws) == 1
    check_raw(small, ws)
    assert header_tag(ws) == 2
    ws[:8] = torch.from_numpy(np.array([2**32 - 2], np.uint64).view(np.uint8)).to(DEV)
    try:
        if withheld is not None:
            lib.pseq_debug_set_wait(1_000_000, withheld)
        cu, info = raw_scan(small, ws)
    finally:
        lib.pseq_debug_set_wait(-1, -1)
    if withheld is None:
        ref_cu, ref_mx = oracle.from_doc_ids(small)
        assert info == (0, len(ref_cu) - 1, ref_mx, small.size)
        np.testing.assert_array_equal(cu[:info[1] + 1].cpu().numpy(), ref_cu)
    else:
        assert info[0] == v._lib.PSEQ_ERR_TIMEOUT
    assert int(ws.count_nonzero()) == 0
    check_raw(big, ws)
    assert header_tag(ws) == 1


def test_doc_ids_random_sequence_of_calls():
    """Sixty calls on the one cached workspace with random shapes (1 to 40
    tiles), kinds and id widths: every call leaves summaries of its own size
    behind, and every later call must ignore them."""
    rng = np.random.default_rng(29)
    kinds = ["runs", "iid", "zeros", "const", "alternating", "long"]
    for i in range(60):
        tiles = int(rng.integers(1, 41))
        B = int(rng.integers(1, 9))
        S = max(1, int(tiles * 16384 // B - rng.integers(0, 4000)))
        dtype = np.int64 if rng.random() < 0.3 else np.int32
        check_doc_ids(synth.random_doc_ids(rng, B, S, kinds[i % len(kinds)], dtype))


def test_doc_ids_graph_replays_share_a_workspace():
    """Two maps captured as CUDA graphs on one workspace and replayed in
    turn: each replay takes the next tag from the header at run time (a
    captured launch carries no tag), so every replay is exact."""
    import ctypes

    v = V()
    lib = v.load_library()
    rng = np.random.default_rng(23)
    maps = [synth.random_doc_ids(rng, 5, 70_000, "runs", np.int32), synth.random_doc_ids(rng, 2, 40_000, "iid", np.int32)]
    refs = [oracle.from_doc_ids(m) for m in maps]
    nbytes = max(lib.pseq_from_doc_ids_workspace_size(*m.shape) for m in maps)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    bufs, graphs = [], []
    for m in maps:
        x = dev(m)
        cu = torch.full((m.size + 1,), -1, dtype=torch.int32, device=DEV)
        info = torch.zeros(32, dtype=torch.uint8, device=DEV)
        bufs.append((x, cu, info))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            assert lib.pseq_from_doc_ids(P(x), 4, m.shape[0], m.shape[1], P(cu), P(info), P(ws), ws.numel(),
                                         ctypes.c_void_p(stream.cuda_stream)) == 0
        graphs.append(g)
    for rep in range(6):
        k = rep % 2
        bufs[k][1].fill_(-1)
        graphs[k].replay()
        torch.cuda.synchronize()
        ref_cu, ref_mx = refs[k]
        assert info_of(bufs[k][2]) == (0, len(ref_cu) - 1, ref_mx, maps[k].size), rep
        np.testing.assert_array_equal(bufs[k][1][: len(ref_cu)].cpu().numpy(), ref_cu)


@pytest.mark.parametrize("withheld", [0, 1, 4])
def test_doc_ids_failed_call_leaves_workspace_usable(withheld):
    """A tile that never publishes (the first, a middle one, the last of
    five): the call reports PSEQ_ERR_TIMEOUT whichever tile waited in vain,
    and the next call on the same buffer is exact."""
    v = V()
    lib = v.load_library()
    rng = np.random.default_rng(22)
    d = synth.random_doc_ids(rng, 4, 20_000, "runs", np.int32)  # 5 tiles
    ws = torch.zeros(lib.pseq_from_doc_ids_workspace_size(*d.shape), dtype=torch.uint8, device=DEV)
    check_raw(d, ws)
    try:
        lib.pseq_debug_set_wait(1_000_000, withheld)
        _, info = raw_scan(d, ws)
    finally:
        lib.pseq_debug_set_wait(-1, -1)
    assert info[0] == v._lib.PSEQ_ERR_TIMEOUT
    check_raw(d, ws)
    check_raw(synth.random_doc_ids(rng, 4, 20_000, "iid", np.int32), ws)


def test_packed_seq_params_api():
    v = V()
    d = torch.tensor([[1, 1, 2, 2, 2, 0]], dtype=torch.int32, device=DEV)
    p = v.packed_seq_params_from_doc_ids(d)
    assert p.cu_seqlens.dtype == torch.int32 and p.cu_seqlens.tolist() == [0, 2, 5, 6]
    assert p.max_seqlen == 3 and p.doc_ids is d
    kw = v.to_flash_attention_kwargs(p)
    assert kw["cu_seq_lens_q"] is kw["cu_seq_lens_k"] is p.cu_seqlens
    assert kw["max_length_q"] == kw["max_length_k"] == 3


# --------------------------------------------------------------------------
# process_input_for_thd / thd_from_batch
# --------------------------------------------------------------------------
def check_thd(batch_np: dict, absorb=True, with_padded=True, hidden=None):
    """Run thd_from_batch on every field of the batch and compare all outputs."""
    v = V()
    real = batch_np["seq_lens"]
    padded = batch_np["seq_lens_padded"] if with_padded else None
    ids = batch_np["input_ids"]
    B, S = ids.shape[:2]
    fields_np = [(ids, 1)]
    if "labels" in batch_np:
        fields_np.append((batch_np["labels"], 1))
    if "position_ids" in batch_np:
        pos = batch_np["position_ids"]
        fields_np.append((pos, pos.shape[0] if pos.ndim == 3 else 1))
    fields_t = [(dev(a), p) for a, p in fields_np]
    if hidden is not None:
        fields_t.append((hidden, 1))
    r = v.thd_from_batch(dev(real), None if padded is None else dev(padded), S, fields_t, -1000, absorb)
    st, n, mx, T = info_of(r["info"])
    try:
        meta = oracle.thd_meta(real, padded, S, -1000, absorb)
    except oracle.OracleValueError:
        assert st == 3, f"device status {st}, oracle raised VALUE"
        return None
    assert st == 0
    assert n == meta["num_sequences"] and T == meta["total_tokens"] and mx == meta["max_seqlen"]
    np.testing.assert_array_equal(r["cu_seqlens"][: n + 1].cpu().numpy(), meta["cu_seqlens"])
    if padded is not None:
        np.testing.assert_array_equal(r["cu_seqlens_padded"][: n + 1].cpu().numpy(), meta["cu_seqlens_padded"])
    assert bool(r["info"][16].item()) == meta["pad_between_seqs"]
    for (a, planes), (dst, _, _) in zip(fields_np, r["dst"]):
        want = oracle.thd_gather(a, meta, B, S, planes=planes)
        got = dst[: want.size].cpu().numpy().reshape(want.shape)
        np.testing.assert_array_equal(got, want)
    if hidden is not None:
        h = hidden.cpu().view(torch.int16).numpy()
        want = oracle.thd_gather(h, meta, B, S)
        got = r["dst"][-1][0][: want.size].cpu().view(torch.int16).numpy().reshape(want.shape)
        np.testing.assert_array_equal(got, want)
    mask_ref = oracle.thd_padding_mask(T, meta["seq_real"], meta["seq_padded"] if padded is not None else None)
    np.testing.assert_array_equal(r["padding_mask"][:T].cpu().numpy(), mask_ref)
    return r


def test_thd_page_example():
    import json
    import os

    with open(os.path.join(os.path.dirname(__file__), "golden", "thd_utils_process_input_example.json")) as f:
        g = json.load(f)
    batch = {k: np.asarray(v, np.int64) for k, v in g["batch"].items()}
    check_thd(batch)
    v = V()
    out = v.process_input_for_thd({k: dev(a) for k, a in batch.items()} | {"qkv_format": "thd"})
    e = g["expected"]
    for k in ("input_ids", "labels", "position_ids", "cu_seqlens", "cu_seqlens_padded"):
        assert out[k].tolist() == e[k], k
    assert int(out["max_seqlen"]) == e["max_seqlen"] and out["max_seqlen"].dtype == torch.int32
    assert out["padding_mask"].tolist() == e["padding_mask"]
    assert out["pad_between_seqs"] == e["pad_between_seqs"]
    assert out["qkv_format"] == "thd"
    assert out["cu_seqlens"].dtype == torch.int32


@pytest.mark.parametrize("seed", range(8))
def test_thd_random(seed):
    rng = np.random.default_rng(500 + seed)
    for trial in range(6):
        B = int(rng.integers(1, 6))
        S = int(rng.integers(1, 3000))
        P = int(rng.integers(1, 40))
        real, padded = synth.random_thd(rng, B, S, P, multiple=int(rng.choice([1, 4, 64])),
                                        interleave_filler=bool(trial % 2), fill_rows=bool(trial % 3 == 0),
                                        with_zero_lengths=True)
        batch = {
            "input_ids": rng.integers(0, 32000, size=(B, S)).astype(np.int64),
            "labels": rng.integers(0, 32000, size=(B, S)).astype(np.int64),
            "position_ids": rng.integers(0, 1 << 40, size=(3, B, S)).astype(np.int64),
            "seq_lens": real,
            "seq_lens_padded": padded,
        }
        H = int(rng.choice([1, 5, 8, 64]))
        hidden = torch.randn(B, S, H, device=DEV).to(torch.bfloat16)
        check_thd(batch, absorb=bool(trial % 2 == 0), with_padded=trial != 5, hidden=hidden)


def test_thd_large_tables_two_kernel_path():
    """B * num_packs above the one-launch limit: metadata kernel + gather."""
    rng = np.random.default_rng(321)
    B, S, P = 48, 700, 60  # 2880 table entries
    real, padded = synth.random_thd(rng, B, S, P, multiple=4, interleave_filler=True)
    batch = {"input_ids": rng.integers(0, 32000, size=(B, S)).astype(np.int64),
             "position_ids": rng.integers(0, 99, size=(3, B, S)).astype(np.int64),
             "seq_lens": real, "seq_lens_padded": padded}
    hidden = torch.randn(B, S, 24, device=DEV).to(torch.bfloat16)
    check_thd(batch, hidden=hidden)
    check_thd(batch, absorb=False, with_padded=False)


@pytest.mark.parametrize("B,P", [(32, 64), (41, 50), (2049, 1)])
def test_thd_at_the_one_launch_table_limit(B, P):
    """Tables of exactly 2048 entries (the one-launch kernel's limit) and of
    2049 and 2050 (the metadata kernel and the gather)."""
    rng = np.random.default_rng(B * 1000 + P)
    S = 96
    real, padded = synth.random_thd(rng, B, S, P, multiple=4, interleave_filler=True)
    batch = {"input_ids": rng.integers(0, 32000, size=(B, S)).astype(np.int64),
             "labels": rng.integers(0, 32000, size=(B, S)).astype(np.int64),
             "seq_lens": real, "seq_lens_padded": padded}
    check_thd(batch)
    check_thd(batch, absorb=False)


def test_thd_many_planes_use_block_copies():
    """More (field, plane) pairs than the row-by-row path takes."""
    rng = np.random.default_rng(99)
    B, S, P = 2, 300, 5
    real, padded = synth.random_thd(rng, B, S, P, multiple=2)
    batch = {"input_ids": rng.integers(0, 32000, size=(B, S)).astype(np.int64),
             "position_ids": rng.integers(0, 99, size=(20, B, S)).astype(np.int64),
             "seq_lens": real, "seq_lens_padded": padded}
    check_thd(batch)


def test_thd_field_widths():
    """1-, 2-, 4- and 8-byte elements with odd row widths (unaligned rows)."""
    rng = np.random.default_rng(42)
    B, S, P = 3, 777, 9
    real, padded = synth.random_thd(rng, B, S, P, multiple=3)
    v = V()
    arrays = [rng.integers(-100, 100, size=(B, S, 3)).astype(np.int8),
              rng.integers(-3000, 3000, size=(B, S, 7)).astype(np.int16),
              rng.integers(-10 ** 9, 10 ** 9, size=(2, B, S, 5)).astype(np.int32),
              rng.integers(-10 ** 12, 10 ** 12, size=(B, S, 3)).astype(np.int64)]
    planes = [1, 1, 2, 1]
    r = v.thd_from_batch(dev(real), dev(padded), S, [(dev(a), p) for a, p in zip(arrays, planes)])
    st, n, mx, T = info_of(r["info"])
    assert st == 0
    meta = oracle.thd_meta(real, padded, S)
    for a, p, (dst, _, _) in zip(arrays, planes, r["dst"]):
        want = oracle.thd_gather(a, meta, B, S, planes=p)
        np.testing.assert_array_equal(dst[: want.size].cpu().numpy().reshape(want.shape), want)


def test_thd_errors():
    cases = [
        (np.array([[3, -1000]]), np.array([[3, 4]])),
        (np.array([[3, 2]]), np.array([[2, 2]])),
        (np.array([[-2, 2]]), np.array([[-2, 2]])),
        (np.array([[5, 3]]), np.array([[5, 4]])),
    ]
    for real, padded in cases:
        batch = {"input_ids": np.arange(8, dtype=np.int64).reshape(1, 8), "seq_lens": real, "seq_lens_padded": padded}
        assert check_thd(batch) is None
    v = V()
    with pytest.raises(ValueError):
        v.process_input_for_thd({"input_ids": dev(np.zeros((1, 8), np.int64)), "seq_lens": dev(cases[1][0]),
                                 "seq_lens_padded": dev(cases[1][1])})


def test_thd_filler_only_and_empty():
    batch = {"input_ids": np.zeros((2, 6), np.int64), "seq_lens": np.full((2, 3), -1000, np.int64),
             "seq_lens_padded": np.full((2, 3), -1000, np.int64)}
    r = check_thd(batch)
    assert info_of(r["info"])[1] == 0


@pytest.mark.parametrize("seed", [0, 1])
def test_thd_small_map_workload(seed):
    c = synth.doc_map_small(seed)
    check_thd({k: c[k] for k in ("input_ids", "labels", "position_ids", "seq_lens", "seq_lens_padded")})


@pytest.mark.parametrize("seed", [0, 1])
def test_thd_ids_workload(seed):
    check_thd(synth.thd_ids(seed))


@pytest.mark.parametrize("H", [128, 200, 2048])
def test_thd_wide_rows_bulk_copy(H):
    """Rows of >= 256 bytes at 16-byte alignment go through the bulk-copy
    engine; check them on ragged layouts, with and without the mask, and as
    chunks of a split batch."""
    rng = np.random.default_rng(H)
    B, S, P = 3, 1500, 20
    real, padded = synth.random_thd(rng, B, S, P, multiple=8, interleave_filler=True)
    batch = {"input_ids": np.zeros((B, S), np.int64), "seq_lens": real, "seq_lens_padded": padded}
    v = V()
    hidden = torch.randn(B, S, H, device=DEV).to(torch.bfloat16)
    r = v.thd_from_batch(dev(real), dev(padded), S, [(hidden, 1)])
    st, n, mx, T = info_of(r["info"])
    meta = oracle.thd_meta(real, padded, S)
    assert st == 0 and T == meta["total_tokens"]
    want = oracle.thd_gather(hidden.cpu().view(torch.int16).numpy(), meta, B, S)
    got = r["dst"][0][0][: T * H].view(torch.int16).cpu().numpy().reshape(T, H)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(r["padding_mask"][:T].cpu().numpy(),
                                  oracle.thd_padding_mask(T, meta["seq_real"], meta["seq_padded"]))
    r2 = v.thd_from_batch(dev(real), dev(padded), S, [(hidden, 1)], want_mask=False)
    np.testing.assert_array_equal(r2["dst"][0][0][: T * H].view(torch.int16).cpu().numpy().reshape(T, H), want)


@pytest.mark.parametrize("gen", ["thd_embeddings", "thd_embeddings_ragged"])
def test_thd_embeddings_workload(gen):
    """bf16 [4, 8192, 4096] at full size: rows that fill S (the stream is the
    batch reshaped) and rows that end short (every row after the first moves
    to a lower stream offset)."""
    c = getattr(synth, gen)(0)
    hidden = c["hidden"].to(DEV)
    v = V()
    B, S, H = hidden.shape
    r = v.thd_from_batch(dev(c["seq_lens"]), dev(c["seq_lens_padded"]), S, [(hidden, 1)])
    st, n, mx, T = info_of(r["info"])
    meta = oracle.thd_meta(c["seq_lens"], c["seq_lens_padded"], S)
    assert st == 0 and n == meta["num_sequences"] and T == meta["total_tokens"] and mx == meta["max_seqlen"]
    np.testing.assert_array_equal(r["cu_seqlens"][: n + 1].cpu().numpy(), meta["cu_seqlens"])
    np.testing.assert_array_equal(r["cu_seqlens_padded"][: n + 1].cpu().numpy(), meta["cu_seqlens_padded"])
    want = oracle.thd_gather(c["hidden"].view(torch.int16).numpy(), meta, B, S)
    got = r["dst"][0][0][: T * H].view(torch.int16).cpu().numpy().reshape(T, H)
    np.testing.assert_array_equal(got, want)
    mask_ref = oracle.thd_padding_mask(T, meta["seq_real"], meta["seq_padded"])
    np.testing.assert_array_equal(r["padding_mask"][:T].cpu().numpy(), mask_ref)


def test_thd_split_calls_match_whole():
    v = V()
    c = synth.thd_ids(3)
    S = c["input_ids"].shape[1]
    m = v.thd_meta(dev(c["seq_lens"]), dev(c["seq_lens_padded"]), S)
    # another conversion of the same size on the same stream in between: the
    # layout thd_gather reads must be the one thd_meta left
    c2 = synth.thd_ids(4)
    v.thd_from_batch(dev(c2["seq_lens"]), dev(c2["seq_lens_padded"]), S, [(dev(c2["input_ids"]), 1)])
    v.thd_meta(dev(c2["seq_lens"]), dev(c2["seq_lens_padded"]), S)
    g = v.thd_gather(m, [(dev(c["input_ids"]), 1)])
    st, n, mx, T = info_of(m["info"])
    meta = oracle.thd_meta(c["seq_lens"], c["seq_lens_padded"], S)
    np.testing.assert_array_equal(g["dst"][0][0][:T].cpu().numpy(), oracle.thd_gather(c["input_ids"], meta, 8, S))


# --------------------------------------------------------------------------
# _thd_padding_mask
# --------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(4))
def test_padding_mask_random(seed):
    v = V()
    rng = np.random.default_rng(900 + seed)
    for _ in range(10):
        n = int(rng.integers(0, 60))
        real = rng.integers(0, 300, size=n).astype(np.int64)
        padded = real + rng.integers(0, 70, size=n).astype(np.int64)
        use_padded = bool(rng.integers(0, 2))
        layout = int((padded if use_padded else real).sum())
        total = layout + int(rng.integers(0, 500))
        mask, info = v.thd_padding_mask(total, dev(real), dev(padded) if use_padded else None)
        st, cnt, mx, tot = info_of(info)
        ref = oracle.thd_padding_mask(total, real, padded if use_padded else None)
        assert st == 0 and cnt == n and tot == total
        np.testing.assert_array_equal(mask.cpu().numpy(), ref)


def test_padding_mask_long_table():
    v = V()
    rng = np.random.default_rng(4)
    n = 3000  # above the one-launch limit
    real = rng.integers(0, 20, size=n).astype(np.int64)
    padded = real + rng.integers(0, 5, size=n).astype(np.int64)
    total = int(padded.sum()) + 77
    mask, info = v.thd_padding_mask(total, dev(real), dev(padded))
    assert info_of(info)[0] == 0
    np.testing.assert_array_equal(mask.cpu().numpy(), oracle.thd_padding_mask(total, real, padded))


def test_padding_mask_errors():
    v = V()
    for real, padded, total in ((np.array([3, 2]), np.array([4, 2]), 5), (np.array([3]), np.array([2]), 9),
                                (np.array([-1]), None, 9)):
        mask, info = v.thd_padding_mask(total, dev(real), None if padded is None else dev(padded))
        assert info_of(info)[0] == 3
        with pytest.raises(oracle.OracleValueError):
            oracle.thd_padding_mask(total, real, padded)


# --------------------------------------------------------------------------
# squeeze
# --------------------------------------------------------------------------
def check_squeeze(prob, multiple, capacity, stretch, width, pad_value=0):
    v = V()
    src = prob["src"]
    N, W = src.shape
    r = v.pack_squeeze(dev(src), dev(prob["real_lens"]), (dev(prob["bin_offsets"]), dev(prob["bin_members"])),
                       multiple, capacity, stretch, width, pad_value)
    st, count, mx, total = info_of(r["info"])
    try:
        ref = oracle.pack_squeeze(src, prob["real_lens"], prob["bin_offsets"], prob["bin_members"], multiple,
                                  capacity, stretch, width, pad_value)
    except oracle.OracleCapacityError:
        assert st == 4
        return None
    except oracle.OracleValueError:
        assert st == 3
        return None
    assert st == 0
    M = int(prob["bin_offsets"][-1])
    nb = len(prob["bin_offsets"]) - 1
    assert count == M and total == ref["max_total"]
    assert mx == (int(prob["real_lens"][prob["bin_members"]].max()) if M else 0)
    np.testing.assert_array_equal(r["packed"].cpu().numpy(), ref["packed"])
    np.testing.assert_array_equal(r["padding_mask"].cpu().numpy(), ref["padding_mask"])
    np.testing.assert_array_equal(r["cu_seqlens"][: M + nb].cpu().numpy(), ref["cu_flat"])
    np.testing.assert_array_equal(r["cu_seqlens_padded"][: M + nb].cpu().numpy(), ref["cu_padded_flat"])
    return r


def test_squeeze_page_example():
    import json
    import os

    with open(os.path.join(os.path.dirname(__file__), "golden", "who_packs_squeeze_example.json")) as f:
        g = json.load(f)
    offs, mem = oracle.bins_to_csr(g["bins"])
    prob = {"src": np.asarray(g["rows"], np.int64), "real_lens": np.asarray(g["input_lengths"], np.int64),
            "bin_offsets": offs, "bin_members": mem}
    check_squeeze(prob, g["multiple"], g["capacity"], False, g["trainer"]["width"])
    check_squeeze(prob, g["multiple"], g["capacity"], True, g["loader"]["width"])
    v = V()
    t = v.squeeze_bins(dev(prob["src"]), dev(prob["real_lens"]), g["bins"], g["multiple"], g["capacity"])
    assert t["packed_input_ids"].tolist() == g["trainer"]["packed"]
    assert t["cu_seqlens"][0].tolist() == g["trainer"]["cu_seqlens"]
    assert t["cu_seqlens_padded"][0].tolist() == g["trainer"]["cu_seqlens_padded"]
    lo = v.squeeze_bins(dev(prob["src"]), dev(prob["real_lens"]), g["bins"], g["multiple"], g["capacity"],
                        stretch_to_capacity=True)
    assert tuple(lo["packed_input_ids"].shape) == (1, g["loader"]["width"])
    assert lo["cu_seqlens_padded"][0].tolist() == g["loader"]["cu_seqlens_padded"]


@pytest.mark.parametrize("dtype", [np.int8, np.int16, np.int32, np.int64])
def test_squeeze_random(dtype):
    rng = np.random.default_rng(77)
    for trial in range(12):
        N = int(rng.integers(1, 40))
        W = int(rng.integers(1, 300))
        prob = synth.random_squeeze(rng, N, W, int(rng.integers(1, 8)), elem_dtype=dtype)
        m = int(rng.choice([1, 3, 8, 64]))
        need = max(sum(-(-int(prob["real_lens"][i]) // m) * m for i in b) for b in prob["bins"])
        stretch = bool(trial % 2)
        cap = need + int(rng.integers(0, 40))
        width = cap if stretch else need + int(rng.integers(0, 5))
        check_squeeze(prob, m, cap, stretch, width, pad_value=int(rng.integers(-5, 5)))


@pytest.mark.parametrize("dtype", [np.int8, np.int16, np.int32, np.int64])
@pytest.mark.parametrize("wide", [False, True])
def test_squeeze_aligned_shapes(dtype, wide):
    # row pitch, width and multiple on 16-byte boundaries: the 16-byte vector
    # path (where the window holds whole vectors), with lengths that end
    # inside a vector and zero-length members
    eb = np.dtype(dtype).itemsize
    V = 16 // eb
    rng = np.random.default_rng(100 + eb + 10 * wide)
    W = 16 * int(rng.integers(8, 40))
    nb, N = (80, 640) if wide else (5, 60)
    prob = synth.random_squeeze(rng, N, W, nb, elem_dtype=dtype)
    for m in (V, 4 * V):
        need = max(sum(-(-int(prob["real_lens"][i]) // m) * m for i in b) for b in prob["bins"])
        width = -(-max(need, 13000 if wide else need + 1) // 16) * 16
        check_squeeze(prob, m, width, True, width, pad_value=-2)
        check_squeeze(prob, m, width + 16, False, width, pad_value=3)


def test_squeeze_many_members():
    rng = np.random.default_rng(8)
    prob = synth.random_squeeze(rng, 1500, 40, 30)
    m = 8
    need = max(sum(-(-int(prob["real_lens"][i]) // m) * m for i in b) for b in prob["bins"])
    check_squeeze(prob, m, need + 16, True, need + 16, pad_value=3)
    check_squeeze(prob, m, need, False, need)


@pytest.mark.parametrize("members", [1, 31, 32, 33, 127, 128, 129, 300])
def test_squeeze_bin_member_counts(members):
    # member counts around a warp and around a round of the block's member
    # scan (256 members per round)
    rng = np.random.default_rng(members)
    prob = synth.random_squeeze(rng, members * 3, 50, 3)
    m = 8
    need = max(sum(-(-int(prob["real_lens"][i]) // m) * m for i in b) for b in prob["bins"])
    check_squeeze(prob, m, need, True, need, pad_value=5)
    one = synth.random_squeeze(rng, members, 50, 1)
    need = sum(-(-int(one["real_lens"][i]) // m) * m for i in one["bins"][0])
    check_squeeze(one, m, need + 64, False, need + 64)


def test_squeeze_bins_denser_than_a_window():
    # multiple 1 and lengths 0..3: a window of output slots meets up to one
    # member per slot, and zero-length members own no slot at all
    rng = np.random.default_rng(9)
    prob = synth.random_squeeze(rng, 6000, 4, 2)
    need = max(sum(int(prob["real_lens"][i]) for i in b) for b in prob["bins"])
    check_squeeze(prob, 1, need, False, need, pad_value=-1)
    check_squeeze(prob, 1, need + 5, True, need + 7, pad_value=2)
    one = synth.random_squeeze(rng, 5000, 2, 1)
    need = int(one["real_lens"].sum())
    check_squeeze(one, 1, need, False, need)


@pytest.mark.parametrize("dtype,m", [(np.int64, 2), (np.int64, 3), (np.int8, 16), (np.int16, 5)])
@pytest.mark.parametrize("bins", [3, 64])
def test_squeeze_window_meets_the_most_members(dtype, m, bins):
    # every member padded to exactly `multiple` slots: a window meets
    # ceil(window / multiple) + 1 members, the most its table is sized for
    # (3 bins: narrow windows; 64 bins: enough CTAs for the wide ones)
    rng = np.random.default_rng(1000 * m + bins)
    per_bin = 16400 // m + 1
    N = bins * per_bin
    info = np.iinfo(dtype)
    prob = {"src": rng.integers(max(info.min, -30000), min(info.max, 30000), size=(N, m)).astype(dtype),
            "real_lens": rng.integers(1, m + 1, size=N).astype(np.int64)}
    perm = rng.permutation(N).astype(np.int32)
    prob["bin_members"] = perm
    prob["bin_offsets"] = (np.arange(bins + 1) * per_bin).astype(np.int32)
    need = per_bin * m
    width = -(-need // 16) * 16
    check_squeeze(prob, m, width, True, width, pad_value=-3)
    check_squeeze(prob, m, need, False, need + 1)


def test_squeeze_wide_windows():
    # enough (window, bin) CTAs that the 16-slot-per-thread kernel runs
    c = synth.squeeze(3, N=2048)
    check_squeeze(c, c["multiple"], c["capacity"], c["stretch"], c["width"], c["pad_value"])
    d = synth.squeeze(4, N=2048, W=1024, multiple=8, capacity=8192)
    check_squeeze(d, d["multiple"], d["capacity"], False, d["capacity"] + 8, pad_value=7)


def bulk_problem(rng, dtype, multiple, width, out_bytes, W=1024):
    """Bins filled greedily from sources of uniform random length (odd and
    zero lengths included) until the output reaches out_bytes."""
    eb = np.dtype(dtype).itemsize
    nb = -(-out_bytes // (width * eb))
    real, bins, n = [], [], 0
    for _ in range(nb):
        members, used = [], 0
        while True:
            r = int(rng.integers(0, W + 1))
            p = -(-r // multiple) * multiple
            if used + p > width - int(rng.integers(0, 3 * multiple)):
                break
            members.append(n)
            real.append(r)
            used += p
            n += 1
        if not members:  # a bin is never empty
            members.append(n)
            real.append(0)
            n += 1
        bins.append(members)
    offs, mem = oracle.bins_to_csr(bins)
    info = np.iinfo(dtype)
    src = rng.integers(max(info.min, -30000), min(info.max, 30000), size=(n, W)).astype(dtype)
    return {"src": src, "real_lens": np.asarray(real, np.int64), "bin_offsets": offs, "bin_members": mem,
            "bins": bins}


@pytest.mark.parametrize("dtype,multiple", [(np.int8, 16), (np.int16, 32), (np.int32, 16), (np.int64, 64)])
def test_squeeze_large_outputs(dtype, multiple):
    """Outputs of 32 MB and more on 16-byte boundaries (the 16-byte vector
    path at its widest grids): runs that end inside 16 bytes, zero lengths,
    hundreds to thousands of bins, stretched and trainer-style rows."""
    eb = np.dtype(dtype).itemsize
    rng = np.random.default_rng(300 + eb)
    width = 16384
    prob = bulk_problem(rng, dtype, multiple, width, 33 << 20)
    check_squeeze(prob, multiple, width, True, width, pad_value=-7)
    check_squeeze(prob, multiple, width + 4096, False, width, pad_value=5)


def test_squeeze_many_windows_unaligned():
    """An odd row pitch (element-wise path) over 700 bins: 2100 window CTAs,
    several waves of them."""
    rng = np.random.default_rng(123)
    m, width = 8, 8002
    prob = bulk_problem(rng, np.int64, m, width, 700 * width * 8, W=301)
    check_squeeze(prob, m, width, True, width, pad_value=-9)
    check_squeeze(prob, m, width + 100, False, width, pad_value=4)


def test_squeeze_large_output_without_mask_and_errors():
    v = V()
    rng = np.random.default_rng(31)
    prob = bulk_problem(rng, np.int64, 64, 32768, 40 << 20)
    src, real = dev(prob["src"]), dev(prob["real_lens"])
    bins = (dev(prob["bin_offsets"]), dev(prob["bin_members"]))
    r = v.pack_squeeze(src, real, bins, 64, 32768, True, 32768, 3, want_mask=False)
    assert r["padding_mask"] is None and info_of(r["info"])[0] == 0
    ref = oracle.pack_squeeze(prob["src"], prob["real_lens"], prob["bin_offsets"], prob["bin_members"], 64, 32768,
                              True, 32768, 3)
    np.testing.assert_array_equal(r["packed"].cpu().numpy(), ref["packed"])
    # a bin over capacity and a member out of range are reported, not copied
    assert check_squeeze(prob, 64, 16384, False, 32768) is None
    bad = dict(prob)
    bad["bin_members"] = prob["bin_members"].copy()
    bad["bin_members"][5] = len(prob["real_lens"]) + 3
    assert check_squeeze(bad, 64, 32768, True, 32768) is None


def test_squeeze_scaled_workload():
    c = synth.squeeze(0, N=16384)
    check_squeeze(c, c["multiple"], c["capacity"], c["stretch"], c["width"], c["pad_value"])


def test_squeeze_workload():
    c = synth.squeeze(0)
    check_squeeze(c, c["multiple"], c["capacity"], c["stretch"], c["width"], c["pad_value"])


def test_squeeze_errors():
    rng = np.random.default_rng(5)
    prob = synth.random_squeeze(rng, 6, 20, 2)
    # capacity too small
    assert check_squeeze(prob, 4, 3, False, 64) is None
    # a member index out of range
    bad = dict(prob)
    bad["bin_members"] = prob["bin_members"].copy()
    bad["bin_members"][0] = 99
    assert check_squeeze(bad, 4, 1000, False, 1000) is None


def test_squeeze_metadata_only_sizes_trainer_row():
    v = V()
    c = synth.squeeze(1)
    r = v.pack_squeeze(dev(c["src"]), dev(c["real_lens"]), (dev(c["bin_offsets"]), dev(c["bin_members"])),
                       c["multiple"], c["capacity"], False, None, 0, with_output=False)
    st, count, mx, total = info_of(r["info"])
    ref = oracle.pack_squeeze(c["src"], c["real_lens"], c["bin_offsets"], c["bin_members"], c["multiple"],
                              c["capacity"], False, c["capacity"])
    assert st == 0 and total == ref["max_total"]

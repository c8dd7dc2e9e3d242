"""Failure detection on the GPU without faulting it.

Every device-side wait in libpseq has a time limit, after which the kernel
reports PSEQ_ERR_TIMEOUT and finishes.  Here one tile is told never to
publish its partial result (the flag nothing sets), the tiles after it run
into a 1 ms limit, and the host reads the status; the context stays usable
and the next call is correct.
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
    yield


def test_lookback_wait_gives_up_and_reports():
    import varlen_attention_metadata_gb300 as v

    lib = v.load_library()
    rng = np.random.default_rng(0)
    d = synth.random_doc_ids(rng, 4, 16384, "runs", np.int32)  # 65536 tokens: five tiles
    dt = torch.from_numpy(d).to(DEV)
    try:
        lib.pseq_debug_set_wait(1_000_000, 1)
        _, info = v.pseq_from_doc_ids(dt)
        assert info[:16].view(torch.int32).tolist()[0] == v._lib.PSEQ_ERR_TIMEOUT
        with pytest.raises(RuntimeError):
            v.check_info(info, "scan")
    finally:
        lib.pseq_debug_set_wait(-1, -1)
    torch.cuda.synchronize()
    p = v.packed_seq_params_from_doc_ids(dt)
    ref_cu, ref_mx = oracle.from_doc_ids(d)
    np.testing.assert_array_equal(p.cu_seqlens.cpu().numpy(), ref_cu)
    assert p.max_seqlen == ref_mx


@pytest.mark.parametrize("withheld", [5, 7])
def test_bridge_wait_gives_up_and_reports(withheld):
    """Chunk 5 (row 1, chunk 1): the row's later chunks run their look-back
    waits out.  Chunk 7 (row 1's last chunk): the row's other chunks run out
    their wait for its summary before filling their shares of the unused
    slots."""
    import varlen_attention_metadata_gb300 as v

    lib = v.load_library()
    rng = np.random.default_rng(1)
    d = synth.random_doc_ids(rng, 2, 4 * 4096, "runs", np.int32)  # 2 rows of 4 chunks
    dt = torch.from_numpy(d).to(DEV)
    try:
        lib.pseq_debug_set_wait(1_000_000, withheld)  # that chunk never publishes
        _, _, _, info = v.pseq_doc_ids_to_lengths(dt, 4 * 4096)
        assert info[:16].view(torch.int32).tolist()[0] == v._lib.PSEQ_ERR_TIMEOUT
    finally:
        lib.pseq_debug_set_wait(-1, -1)
    torch.cuda.synchronize()
    # the workspace is clean again: the next call is exact
    real, padded, pos, info = v.pseq_doc_ids_to_lengths(dt, 4 * 4096)
    ref = oracle.doc_ids_to_lengths(d, 4 * 4096)
    assert info[:16].view(torch.int32).tolist()[0] == 0
    np.testing.assert_array_equal(real.cpu().numpy(), ref["seq_lens"])
    np.testing.assert_array_equal(padded.cpu().numpy(), ref["seq_lens_padded"])
    np.testing.assert_array_equal(pos.cpu().numpy(), ref["position_ids"])


def test_host_side_errors_launch_nothing():
    import varlen_attention_metadata_gb300 as v

    lib = v.load_library()
    before = lib.pseq_launch_count()
    d = torch.zeros(2, 8, dtype=torch.int32, device=DEV)
    cu = torch.empty(17, dtype=torch.int32, device=DEV)
    info = torch.empty(4, dtype=torch.int32, device=DEV)
    import ctypes

    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.pseq_from_doc_ids(p(d), 4, 2, 8, p(cu), p(info), None, 0, None)
    assert st == v._lib.PSEQ_ERR_ARG and "workspace" in v._lib.last_error()
    ws = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    st = lib.pseq_from_doc_ids(ctypes.c_void_p(d.data_ptr() + 2), 4, 2, 8, p(cu), p(info), p(ws), 4096, None)
    assert st == v._lib.PSEQ_ERR_ARG and "misaligned" in v._lib.last_error()
    st = lib.pseq_from_doc_ids(p(d), 4, 1 << 20, 1 << 20, p(cu), p(info), p(ws), 4096, None)
    assert st == v._lib.PSEQ_ERR_OVERFLOW
    assert lib.pseq_launch_count() == before
    with pytest.raises(TypeError):
        v.pseq_from_doc_ids(torch.zeros(2, 2, dtype=torch.float32, device=DEV))
    with pytest.raises(ValueError):
        v.pseq_from_doc_ids(torch.zeros(2, 2, dtype=torch.int32))  # CPU tensor: no CPU path


def test_outputs_stay_inside_their_buffers():
    """Guard bands around every output of the THD conversion."""
    import varlen_attention_metadata_gb300 as v

    c = synth.thd_ids(5)
    B, S = c["input_ids"].shape
    r = v.thd_from_batch(torch.from_numpy(c["seq_lens"]).to(DEV), torch.from_numpy(c["seq_lens_padded"]).to(DEV), S,
                         [(torch.from_numpy(c["input_ids"]).to(DEV), 1)])
    # thd_from_batch allocates exact worst-case buffers; re-run into guarded ones through the C ABI
    lib = v.load_library()
    import ctypes

    P = c["seq_lens"].shape[1]
    g = 32
    ids = torch.from_numpy(c["input_ids"]).to(DEV)
    dst = torch.full((B * S + 2 * g,), -7, dtype=torch.int64, device=DEV)
    mask = torch.full((B * S + 2 * g,), 0x5A, dtype=torch.uint8, device=DEV)
    cu = torch.full((B * P + 1 + 2 * g,), -9, dtype=torch.int32, device=DEV)
    cup = torch.full((B * P + 1 + 2 * g,), -9, dtype=torch.int32, device=DEV)
    info = torch.zeros(8, dtype=torch.int32, device=DEV)
    ws = torch.empty(lib.thd_workspace_size(B, P), dtype=torch.uint8, device=DEV)
    f = (v._lib.PseqField * 1)()
    f[0].src = ids.data_ptr()
    f[0].dst = dst.data_ptr() + 8 * g
    f[0].elem_bytes = 8
    f[0].planes = 1
    f[0].row_elems = 1
    p = lambda t, off=0: ctypes.c_void_p(t.data_ptr() + off)
    real = torch.from_numpy(c["seq_lens"]).to(DEV)
    padded = torch.from_numpy(c["seq_lens_padded"]).to(DEV)
    st = lib.thd_from_batch(p(real), p(padded), B, S, P, -1000, 1, f, 1, p(cu, 4 * g), p(cup, 4 * g), p(mask, g),
                            p(info, 16), p(info), p(ws), ws.numel(), None)
    assert st == 0
    s, n, mx, T = info[:4].tolist()
    assert s == 0
    d = dst.cpu().numpy()
    assert np.all(d[:g] == -7) and np.all(d[g + T:] == -7)
    m = mask.cpu().numpy()
    assert np.all(m[:g] == 0x5A) and np.all(m[g + T:] == 0x5A)
    for arr in (cu, cup):
        a = arr.cpu().numpy()
        assert np.all(a[:g] == -9) and np.all(a[g + n + 1:] == -9)
    meta = oracle.thd_meta(c["seq_lens"], c["seq_lens_padded"], S)
    np.testing.assert_array_equal(d[g:g + T], oracle.thd_gather(c["input_ids"], meta, B, S))

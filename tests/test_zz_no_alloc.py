"""pseq_from_doc_ids_static: the doc_ids scan for callers that cannot
allocate device memory when they call in (a memory pool that forbids new
allocations, a plugin handed only input and output pointers, a process that
reserved all of HBM).  Its scratch is a static device array inside
libpseq.so, shared by every call.

Every case is called twice in a row through the C ABI and compared with the
oracle and with the workspace-taking pseq_from_doc_ids on the same input
(bit-exact: the work is integer).  The maps run from one tile to exactly
PSEQ_STATIC_MAX_TOKENS tokens, which uses the array's last slot.  Collected
last, so a run that stops at the first failure has run every other test
first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from varlen_attention_metadata_gb300 import _lib, build

    build.build()
    return _lib.load()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _static(lib, ids, B, S):
    cu = torch.full((B * S + 1,), -1, dtype=torch.int32, device=DEV)
    info = torch.zeros(4, dtype=torch.int32, device=DEV)
    assert lib.pseq_from_doc_ids_static(_p(ids), ids.element_size(), B, S, _p(cu), _p(info), _stream()) == 0
    return cu, info


def _run_both(lib, d: np.ndarray):
    B, S = d.shape
    ids = torch.from_numpy(d).to(DEV)
    cu_a = torch.full((B * S + 1,), -1, dtype=torch.int32, device=DEV)
    info_a = torch.zeros(4, dtype=torch.int32, device=DEV)
    ws = torch.zeros(lib.pseq_from_doc_ids_workspace_size(B, S), dtype=torch.uint8, device=DEV)
    assert lib.pseq_from_doc_ids(_p(ids), ids.element_size(), B, S, _p(cu_a), _p(info_a), _p(ws), ws.numel(),
                                 _stream()) == 0
    ref_cu, ref_mx = oracle.from_doc_ids(d)
    n = len(ref_cu) - 1
    for _ in range(2):  # the second call finds the array as the first left it
        cu_b, info_b = _static(lib, ids, B, S)
        torch.cuda.synchronize()
        ia, ib = info_a.tolist(), info_b.tolist()
        assert ib == [0, n, ref_mx, B * S] and ia == ib
        np.testing.assert_array_equal(cu_b[: n + 1].cpu().numpy(), ref_cu)
        assert torch.equal(cu_a[: n + 1], cu_b[: n + 1])
        assert torch.all(cu_b[n + 1:] == -1)  # nothing written past the boundaries


def test_static_scratch_matches_oracle_and_workspace_call_twice(lib):
    rng = np.random.default_rng(21)
    _run_both(lib, synth.doc_map_stress(3))                              # 2M tokens, ~258k segments
    _run_both(lib, synth.random_doc_ids(rng, 3, 5001, "runs", np.int64))  # int64 ids
    _run_both(lib, synth.random_doc_ids(rng, 1, 9000, "runs", np.int32))  # one tile


def test_static_scratch_at_its_token_limit(lib):
    from varlen_attention_metadata_gb300 import _lib

    B, S = 512, _lib.PSEQ_STATIC_MAX_TOKENS // 512  # exactly the limit: every slot of the array in use
    _run_both(lib, synth.doc_map_stress(5, B=B, S=S))


def test_static_scratch_recovers_after_a_timed_out_call(lib):
    """A call whose look-back waits run out (one tile withholds its summary)
    reports PSEQ_ERR_TIMEOUT; the next call clears the array and is exact."""
    from varlen_attention_metadata_gb300 import _lib

    d = synth.random_doc_ids(np.random.default_rng(8), 4, 16384, "runs", np.int32)  # 5 tiles
    ids = torch.from_numpy(d).to(DEV)
    try:
        lib.pseq_debug_set_wait(1_000_000, 2)  # 1 ms limit; tile 2 never publishes
        _, info = _static(lib, ids, *d.shape)
        torch.cuda.synchronize()
        assert info.tolist()[0] == _lib.PSEQ_ERR_TIMEOUT
    finally:
        lib.pseq_debug_set_wait(-1, -1)
    _run_both(lib, d)


def test_static_scratch_rejects_oversized_maps(lib):
    from varlen_attention_metadata_gb300 import _lib

    before = lib.pseq_launch_count()
    big_s = _lib.PSEQ_STATIC_MAX_TOKENS // 2 + 1
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check fails first
    st = lib.pseq_from_doc_ids_static(fake, 4, 2, big_s, fake, fake, None)
    assert st == _lib.PSEQ_ERR_ARG
    assert "static scratch limit" in _lib.last_error()
    assert lib.pseq_launch_count() == before

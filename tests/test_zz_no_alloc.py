"""pseq_from_doc_ids_static: the doc_ids scan for callers that cannot
allocate device memory when they call in (a memory pool that forbids new
allocations, a plugin handed only input and output pointers, a process that
reserved all of HBM).  Its scratch is a static device array inside
libpseq.so, shared by every call.

Called twice in a row through the C ABI, each time against the
workspace-taking pseq_from_doc_ids on the same input (bit-exact: the work is
integer).  Collected last, so a run that stops at the first failure has run
every other test first; it also passes alone in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

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


def _run_both(lib, d: np.ndarray):
    B, S = d.shape
    ids = torch.from_numpy(d).to(DEV)
    eb = ids.element_size()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    cu_a = torch.full((B * S + 1,), -1, dtype=torch.int32, device=DEV)
    info_a = torch.zeros(4, dtype=torch.int32, device=DEV)
    ws = torch.zeros(lib.pseq_from_doc_ids_workspace_size(B, S), dtype=torch.uint8, device=DEV)
    assert lib.pseq_from_doc_ids(_p(ids), eb, B, S, _p(cu_a), _p(info_a), _p(ws), ws.numel(), stream) == 0
    cu_b = torch.full((B * S + 1,), -1, dtype=torch.int32, device=DEV)
    info_b = torch.zeros(4, dtype=torch.int32, device=DEV)
    assert lib.pseq_from_doc_ids_static(_p(ids), eb, B, S, _p(cu_b), _p(info_b), stream) == 0
    torch.cuda.synchronize()
    ia, ib = info_a.tolist(), info_b.tolist()
    assert ia[0] == 0 and ib == ia
    n = ia[1]
    assert torch.equal(cu_a[: n + 1], cu_b[: n + 1])
    assert torch.all(cu_b[n + 1:] == -1)  # nothing written past the boundaries


def test_static_scratch_matches_workspace_call_twice(lib):
    rng = np.random.default_rng(21)
    _run_both(lib, synth.doc_map_stress(3))                              # 512 tiles, ~258k segments
    _run_both(lib, synth.random_doc_ids(rng, 3, 5001, "runs", np.int64))  # fewer tiles, int64 ids


def test_static_scratch_rejects_oversized_maps(lib):
    from varlen_attention_metadata_gb300 import _lib

    before = lib.pseq_launch_count()
    big_s = _lib.PSEQ_STATIC_MAX_TOKENS // 2 + 1
    fake = ctypes.c_void_p(256)  # never dereferenced: the size check fails first
    st = lib.pseq_from_doc_ids_static(fake, 4, 2, big_s, fake, fake, None)
    assert st == _lib.PSEQ_ERR_ARG
    assert "static scratch limit" in _lib.last_error()
    assert lib.pseq_launch_count() == before

"""The C ABI library builds, loads and exports every entry point declared in
include/pseq.h; host-side argument checks answer without a GPU (no compute
call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    with open(os.path.join(ROOT, "include", "pseq.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([a-z_][a-z0-9_]*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "while", "sizeof")))


@pytest.fixture(scope="module")
def lib():
    from varlen_attention_metadata_gb300 import build, _lib

    build.build()
    return _lib.load()


def test_header_declares_the_hot_path():
    names = declared_functions()
    for want in ("pseq_from_doc_ids", "thd_from_batch", "thd_padding_mask", "pack_squeeze", "thd_meta",
                 "thd_gather"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    from varlen_attention_metadata_gb300 import _lib

    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert set(names) == set(_lib.SIGNATURES), set(names) ^ set(_lib.SIGNATURES)


def test_workspace_sizes(lib):
    assert lib.pseq_from_doc_ids_workspace_size(-1, 4) == 0
    assert lib.pseq_from_doc_ids_workspace_size(1 << 20, 1 << 20) == 0  # B*S over INT32_MAX
    small = lib.pseq_from_doc_ids_workspace_size(4, 2048)
    big = lib.pseq_from_doc_ids_workspace_size(64, 32768)
    assert 0 < small < big
    assert lib.thd_workspace_size(8, 64) >= 8 * 64 * 16
    # the squeeze's scratch is a fixed header (a counter and running totals)
    assert lib.pack_squeeze_workspace_size(256, 8) > 0
    assert lib.pack_squeeze_workspace_size(16384, 65535) == lib.pack_squeeze_workspace_size(256, 8)


def test_host_argument_errors_without_gpu(lib):
    from varlen_attention_metadata_gb300 import _lib

    P = ctypes.c_void_p
    fake = P(0x1000)  # never dereferenced: every call below fails its host checks first
    assert lib.pseq_from_doc_ids(None, 4, -1, 2, None, None, None, 0, None) == _lib.PSEQ_ERR_ARG
    assert lib.pseq_from_doc_ids(fake, 3, 2, 2, fake, fake, fake, 1 << 20, None) == _lib.PSEQ_ERR_ARG
    assert lib.pseq_from_doc_ids(fake, 4, 1 << 20, 1 << 20, fake, fake, fake, 1 << 20, None) == _lib.PSEQ_ERR_OVERFLOW
    assert "INT32_MAX" in _lib.last_error()
    assert lib.thd_from_batch(fake, None, -1, 4, 4, -1000, 1, None, 0, fake, None, None, None, fake, fake, 0,
                              None) == _lib.PSEQ_ERR_ARG
    assert lib.thd_meta(fake, None, 2, 4, 4, -1000, 1, None, None, None, fake, fake, 1 << 20,
                        None) == _lib.PSEQ_ERR_ARG
    assert lib.thd_gather(None, 9, 2, 4, 4, None, fake, 1 << 20, None) == _lib.PSEQ_ERR_ARG
    assert lib.thd_padding_mask(-1, None, None, 0, None, None, None, 0, None) == _lib.PSEQ_ERR_ARG
    assert lib.pack_squeeze(fake, 2, 2, 3, fake, fake, fake, 1, 2, 4, 8, 0, 8, 0, fake, fake, fake, fake, fake,
                            fake, 1 << 20, None) == _lib.PSEQ_ERR_ARG
    assert lib.pack_squeeze(fake, 2, 2, 8, fake, fake, fake, 1, 2, 0, 8, 0, 8, 0, fake, fake, fake, fake, fake,
                            fake, 1 << 20, None) == _lib.PSEQ_ERR_ARG
    assert lib.pack_squeeze(fake, 2, 2, 8, fake, fake, fake, 1, 2, 4, 16, 1, 8, 0, fake, fake, fake, fake, fake,
                            fake, 1 << 20, None) == _lib.PSEQ_ERR_ARG  # stretch needs width >= capacity
    # size limits
    assert lib.pack_squeeze(fake, 2, 2, 8, fake, fake, fake, 1, 2, 4, 8, 0, 2**31 - 65535, 0, fake, fake, fake, fake,
                            fake, fake, 1 << 20, None) == _lib.PSEQ_ERR_OVERFLOW  # width past 2^31 - 2^16
    assert lib.pack_squeeze(fake, 2, 2, 8, fake, fake, fake, 65536, 65536, 4, 8, 0, 8, 0, fake, fake, fake, fake,
                            fake, fake, 1 << 20, None) == _lib.PSEQ_ERR_ARG  # more bins than the grid holds
    assert lib.thd_mask_from_token_ids(fake, 4, 2**31, 0, fake, fake, fake, 1 << 20, None) == _lib.PSEQ_ERR_OVERFLOW
    assert lib.pack_ffd(fake, 8193, 1, 100, fake, fake, fake, None) == _lib.PSEQ_ERR_ARG
    assert lib.pseq_doc_ids_to_lengths(fake, 4, 1, 2**31 - 4000, 4, -1000, fake, fake, None, fake, fake, 1 << 20,
                                       None) == _lib.PSEQ_ERR_OVERFLOW  # one row within a chunk of INT32_MAX
    assert lib.pseq_version() >= 100


def test_debug_wait_limit_is_clamped(lib):
    """No setting lifts the bound on device-side waits: a limit above the
    1 s default is clamped to it, a negative one restores it."""
    try:
        lib.pseq_debug_set_wait(2**63 - 1, 5)
        assert lib.pseq_debug_wait_limit_ns() == 1_000_000_000
        lib.pseq_debug_set_wait(1_000_000, -1)
        assert lib.pseq_debug_wait_limit_ns() == 1_000_000
        lib.pseq_debug_set_wait(0, -1)
        assert lib.pseq_debug_wait_limit_ns() == 0
        lib.pseq_debug_set_wait(-7, -1)
        assert lib.pseq_debug_wait_limit_ns() == 1_000_000_000
    finally:
        lib.pseq_debug_set_wait(-1, -1)
    assert lib.pseq_debug_wait_limit_ns() == 1_000_000_000


def test_product_path_refuses_cpu_tensors():
    import torch

    import varlen_attention_metadata_gb300 as v

    with pytest.raises(ValueError, match="CUDA"):
        v.pseq_from_doc_ids(torch.zeros(2, 3, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA"):
        v.process_input_for_thd({"input_ids": torch.zeros(1, 4, dtype=torch.int64),
                                 "seq_lens": torch.tensor([[4]])})


def test_missing_library_fails_loudly(tmp_path):
    from varlen_attention_metadata_gb300 import _lib

    with pytest.raises(RuntimeError, match="no fallback"):
        _lib.load(str(tmp_path / "libpseq.so"))


def test_product_package_does_not_import_the_oracle():
    pkg = os.path.join(ROOT, "varlen_attention_metadata_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    text = fh.read()
                assert not re.search(r"\bimport oracle\b|\bfrom oracle\b|pseq_oracle", text), f

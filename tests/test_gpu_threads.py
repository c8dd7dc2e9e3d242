"""Several host threads calling the library at once, each on its own CUDA
stream.

The host runtime fills its per-device caches (SM count, occupancy, shared
memory attributes) under locks and keeps error text per thread, and the
binding hands every (kind, device, stream) its own workspace.  Four threads
interleave doc_ids scans, THD conversions (narrow fields and wide rows) and
squeezes on their own streams; every result is checked against the oracle.
"""
import threading

import numpy as np
import pytest
import torch

import oracle
import synth

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def built():
    from varlen_attention_metadata_gb300 import build

    build.build()
    yield


def info_of(t):
    return t[:16].view(torch.int32).tolist()[:4] if t.dtype == torch.uint8 else t[:4].tolist()


def calls(seed: int, rounds: int):
    import varlen_attention_metadata_gb300 as v

    rng = np.random.default_rng(seed)
    for it in range(rounds):
        # doc_ids scan over several tiles
        d = synth.random_doc_ids(rng, 3, 20000 + 97 * it, "runs", np.int32)
        p = v.packed_seq_params_from_doc_ids(torch.from_numpy(d).to(DEV))
        ref_cu, ref_mx = oracle.from_doc_ids(d)
        np.testing.assert_array_equal(p.cu_seqlens.cpu().numpy(), ref_cu)
        assert p.max_seqlen == ref_mx
        # THD conversion: narrow ids and wide bf16 rows (the bulk-copy kernel)
        B, S, P = 3, 700 + it, 12
        real, padded = synth.random_thd(rng, B, S, P, multiple=8, interleave_filler=True)
        ids = rng.integers(0, 32000, size=(B, S)).astype(np.int64)
        hidden = torch.randn(B, S, 256, device=DEV).to(torch.bfloat16)
        meta = oracle.thd_meta(real, padded, S)
        T = meta["total_tokens"]
        r = v.thd_from_batch(torch.from_numpy(real).to(DEV), torch.from_numpy(padded).to(DEV), S,
                             [(torch.from_numpy(ids).to(DEV), 1)])
        assert info_of(r["info"])[0] == 0
        np.testing.assert_array_equal(r["dst"][0][0][:T].cpu().numpy(), oracle.thd_gather(ids, meta, B, S))
        np.testing.assert_array_equal(r["padding_mask"][:T].cpu().numpy(),
                                      oracle.thd_padding_mask(T, meta["seq_real"], meta["seq_padded"]))
        r = v.thd_from_batch(torch.from_numpy(real).to(DEV), torch.from_numpy(padded).to(DEV), S, [(hidden, 1)])
        assert info_of(r["info"])[0] == 0
        want = oracle.thd_gather(hidden.cpu().view(torch.int16).numpy(), meta, B, S)
        np.testing.assert_array_equal(r["dst"][0][0][: T * 256].view(torch.int16).cpu().numpy().reshape(T, 256), want)
        # squeeze into bins
        c = synth.squeeze(seed * 10 + it, N=24, W=300, multiple=16, capacity=2048)
        dv = lambda a: torch.from_numpy(a).to(DEV)  # noqa: E731
        q = v.pack_squeeze(dv(c["src"]), dv(c["real_lens"]), (dv(c["bin_offsets"]), dv(c["bin_members"])),
                           c["multiple"], c["capacity"], c["stretch"], c["width"], c["pad_value"])
        ref = oracle.pack_squeeze(c["src"], c["real_lens"], c["bin_offsets"], c["bin_members"], c["multiple"],
                                  c["capacity"], c["stretch"], c["width"], c["pad_value"])
        assert info_of(q["info"])[0] == 0
        np.testing.assert_array_equal(q["packed"].cpu().numpy(), ref["packed"])
        np.testing.assert_array_equal(q["padding_mask"].cpu().numpy(), ref["padding_mask"])


def test_threads_on_their_own_streams():
    errors = []

    def worker(seed):
        try:
            torch.cuda.set_device(DEV)
            stream = torch.cuda.Stream(DEV)
            with torch.cuda.stream(stream):
                calls(seed, rounds=4)
        except Exception as e:  # reported to the main thread below
            errors.append(f"thread {seed}: {e!r}")

    threads = [threading.Thread(target=worker, args=(seed,)) for seed in range(1, 5)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=600)
    assert not any(t.is_alive() for t in threads), "a worker thread did not finish"
    assert not errors, errors

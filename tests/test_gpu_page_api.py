"""The pages' functions with 3D embeddings, through the product binding.

[thd_utils] process_input_for_thd takes input_ids as token ids [B, S] or, in
pipeline-parallel stages, embeddings [B, S, H], and returns input_ids as
[total_tokens, H] for the latter; split_batch_into_thd_chunks does the same
per chunk and stacks the chunks.  Here bf16 embeddings go through both
functions with 2D and mRoPE positions, on layouts whose rows fill S and on
layouts whose rows end short, and every returned tensor is compared element
by element with the oracle (bf16 values compared as their 16-bit patterns).
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


def V():
    import varlen_attention_metadata_gb300 as v

    return v


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).to(DEV)


def bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a tensor; bf16 as its int16 bit patterns."""
    t = t.cpu()
    return t.view(torch.int16).numpy() if t.dtype == torch.bfloat16 else t.numpy()


def make_batch(rng, B, S, H, P, mrope, fill_rows, multiple=8):
    real, padded = synth.random_thd(rng, B, S, P, multiple=multiple, fill_rows=fill_rows)
    hidden = torch.from_numpy(rng.standard_normal((B, S, H), dtype=np.float32)).to(torch.bfloat16)
    pos = (rng.integers(0, 1 << 20, size=(3, B, S)) if mrope else rng.integers(0, 1 << 20, size=(B, S)))
    host = {"input_ids": hidden.view(torch.int16).numpy(),
            "labels": rng.integers(0, 32000, size=(B, S)).astype(np.int64),
            "position_ids": pos.astype(np.int64), "seq_lens": real, "seq_lens_padded": padded}
    gpu = {"input_ids": hidden.to(DEV), "labels": dev(host["labels"]), "position_ids": dev(host["position_ids"]),
           "seq_lens": dev(real), "seq_lens_padded": dev(padded), "qkv_format": "thd"}
    return host, gpu


@pytest.mark.parametrize("H", [64, 128, 4096])
@pytest.mark.parametrize("mrope", [False, True])
@pytest.mark.parametrize("fill_rows", [True, False])
def test_process_input_for_thd_embeddings(H, mrope, fill_rows):
    rng = np.random.default_rng(H + 10 * mrope + 100 * fill_rows)
    B, S = 3, 700
    host, gpu = make_batch(rng, B, S, H, 12, mrope, fill_rows)
    out = V().process_input_for_thd(gpu)
    ref = oracle.process_input_for_thd(host)
    T = ref["total_tokens"]
    assert out["input_ids"].shape == (T, H) and out["input_ids"].dtype == torch.bfloat16
    assert out["labels"].shape == (T,)
    assert out["position_ids"].shape == ((3, 1, T) if mrope else (T,))
    assert out["padding_mask"].shape == (T,) and out["padding_mask"].dtype == torch.bool
    for k in ("input_ids", "labels", "position_ids", "cu_seqlens", "cu_seqlens_padded", "padding_mask"):
        np.testing.assert_array_equal(bits(out[k]), ref[k], err_msg=k)
    assert int(out["max_seqlen"]) == ref["max_seqlen"]
    assert out["pad_between_seqs"] == ref["pad_between_seqs"]
    assert out["qkv_format"] == "thd"


def test_process_input_for_thd_embeddings_only():
    """Embeddings as the only field: the bulk-copy path of the library."""
    rng = np.random.default_rng(5)
    B, S, H = 2, 1024, 2048
    real, padded = synth.random_thd(rng, B, S, 16, multiple=16)
    hidden = torch.from_numpy(rng.standard_normal((B, S, H), dtype=np.float32)).to(torch.bfloat16)
    out = V().process_input_for_thd({"input_ids": hidden.to(DEV), "seq_lens": dev(real),
                                     "seq_lens_padded": dev(padded)})
    ref = oracle.process_input_for_thd({"input_ids": hidden.view(torch.int16).numpy(), "seq_lens": real,
                                        "seq_lens_padded": padded})
    assert out["input_ids"].shape == (ref["total_tokens"], H)
    np.testing.assert_array_equal(bits(out["input_ids"]), ref["input_ids"])
    np.testing.assert_array_equal(bits(out["padding_mask"]), ref["padding_mask"])


def equal_chunk_lengths(rng, B, S, P, num_chunks, short):
    """Lengths whose chunks all produce streams of one length T; with `short`
    the rows end before S, so T is less than the chunk's B/num_chunks * S."""
    Bc = B // num_chunks
    room = S - (S // 4 if short else 0)
    real = np.full((B, P), -1000, np.int64)
    padded = np.full((B, P), -1000, np.int64)
    for c in range(num_chunks):
        for b in range(c * Bc, (c + 1) * Bc):
            # the same row totals in every chunk, cut differently
            cuts = np.sort(rng.choice(np.arange(1, room), size=min(P - 1, 3), replace=False))
            pl = np.diff(np.concatenate([[0], cuts, [room]]))
            for k, x in enumerate(pl):
                padded[b, k] = x
                real[b, k] = int(rng.integers(0, x + 1))
    return real, padded


@pytest.mark.parametrize("mrope", [False, True])
@pytest.mark.parametrize("short", [False, True])
def test_split_batch_into_thd_chunks_embeddings(mrope, short):
    rng = np.random.default_rng(7 + mrope + 2 * short)
    B, S, H, P, nc = 4, 640, 256, 6, 2
    real, padded = equal_chunk_lengths(rng, B, S, P, nc, short)
    hidden = torch.from_numpy(rng.standard_normal((B, S, H), dtype=np.float32)).to(torch.bfloat16)
    pos = rng.integers(0, 1 << 20, size=(3, B, S) if mrope else (B, S)).astype(np.int64)
    labels = rng.integers(0, 32000, size=(B, S)).astype(np.int64)
    host = {"input_ids": hidden.view(torch.int16).numpy(), "labels": labels, "position_ids": pos,
            "seq_lens": real, "seq_lens_padded": padded}
    gpu = {"input_ids": hidden.to(DEV), "labels": dev(labels), "position_ids": dev(pos), "seq_lens": dev(real),
           "seq_lens_padded": dev(padded)}
    out = V().split_batch_into_thd_chunks(gpu, nc)
    ref = oracle.split_batch_into_thd_chunks(host, nc)
    T = ref["input_ids"].shape[1]
    assert T == (B // nc) * S - (S // 4 if short else 0) * (B // nc)
    assert out["input_ids"].shape == (nc, T, H) and out["input_ids"].dtype == torch.bfloat16
    assert out["labels"].shape == (nc, T)
    assert out["position_ids"].shape == ((nc, 3, 1, T) if mrope else (nc, T))
    assert out["padding_mask"].shape == (nc, T)
    for k in ("input_ids", "labels", "position_ids", "padding_mask", "cu_seqlens", "cu_seqlens_padded"):
        np.testing.assert_array_equal(bits(out[k]), ref[k], err_msg=k)
    np.testing.assert_array_equal(out["max_seqlen"].cpu().numpy(), ref["max_seqlen"])
    np.testing.assert_array_equal(out["pad_between_seqs"].cpu().numpy(), ref["pad_between_seqs"])

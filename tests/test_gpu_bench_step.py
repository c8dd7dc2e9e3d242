"""The step exactly as bench.py times it, checked against the oracle.

bench.py issues the five workloads' calls from prebuilt ctypes arguments, the
embedding conversion first on the step's stream and the other calls beside it
on a second stream, step after step on the same buffers and workspaces.  These tests run that object
(``bench.NativeStep``) and compare every output of every call with the oracle
element by element, after two-stream steps and after a one-stream step.
"""
import os
import sys

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module")
def step():
    import bench
    from varlen_attention_metadata_gb300 import build

    build.build()
    host = bench.make_inputs(0)
    stream = torch.cuda.Stream(DEV)
    side = torch.cuda.Stream(DEV)
    s = bench.NativeStep(host, DEV, stream, side_stream=side)
    with torch.cuda.stream(stream):
        s.run()
    s.resolve()
    return s


def info_of(t):
    return t[:4].tolist()


def check_outputs(s):
    torch.cuda.synchronize(DEV)
    h = s.host
    for name, get in s._finish.items():
        res = get()
        info = info_of(res[0])
        assert info[0] == 0, (name, info)
        if name.startswith("map"):
            _, cu, _ = res
            ref_cu, ref_mx = oracle.from_doc_ids(h[name])
            assert info[1] == len(ref_cu) - 1 and info[2] == ref_mx
            np.testing.assert_array_equal(cu[: info[1] + 1].cpu().numpy(), ref_cu)
        elif name == "thd_emb":
            _, cu, cup, mask, dsts = res
            emb = h[name]
            hid = emb["hidden"].view(torch.int16).numpy()
            meta = oracle.thd_meta(emb["seq_lens"], emb["seq_lens_padded"], hid.shape[1])
            n, T = meta["num_sequences"], meta["total_tokens"]
            assert info[1] == n and info[3] == T and info[2] == meta["max_seqlen"]
            np.testing.assert_array_equal(cu[: n + 1].cpu().numpy(), meta["cu_seqlens"])
            np.testing.assert_array_equal(cup[: n + 1].cpu().numpy(), meta["cu_seqlens_padded"])
            ref_mask = oracle.thd_padding_mask(T, meta["seq_real"], meta["seq_padded"])
            np.testing.assert_array_equal(mask[:T].cpu().numpy().astype(bool), ref_mask)
            dst, planes, row, eb = dsts[0]
            got = dst[: T * row].view(torch.int16).cpu().numpy().reshape(T, row)
            # compare row by row against the source rows the layout names
            seq_of_row = np.repeat(np.arange(n), meta["seq_padded"])
            within = np.arange(T) - np.repeat(meta["cu_seqlens_padded"][:-1], meta["seq_padded"])
            src_b = meta["seq_row"][seq_of_row]
            src_s = meta["seq_off"][seq_of_row] + within
            np.testing.assert_array_equal(got, hid[src_b, src_s])
        elif name.startswith("thd"):
            _, cu, cup, mask, dsts = res
            bt = h[name]
            ref = oracle.process_input_for_thd(
                {k: bt[k] for k in ("input_ids", "labels", "position_ids", "seq_lens", "seq_lens_padded")})
            T = ref["total_tokens"]
            n = len(ref["cu_seqlens"]) - 1
            assert info[1] == n and info[3] == T and info[2] == ref["max_seqlen"]
            np.testing.assert_array_equal(cu[: n + 1].cpu().numpy(), ref["cu_seqlens"])
            np.testing.assert_array_equal(cup[: n + 1].cpu().numpy(), ref["cu_seqlens_padded"])
            np.testing.assert_array_equal(mask[:T].cpu().numpy().astype(bool), ref["padding_mask"])
            for (dst, planes, row, eb), key in zip(dsts, ("input_ids", "labels", "position_ids")):
                got = dst[: planes * T].cpu().numpy()
                np.testing.assert_array_equal(got, ref[key].reshape(-1))
        else:
            _, cu, cup, mask, out, ncu = res
            c = h[name]
            ref = oracle.pack_squeeze(c["src"], c["real_lens"], c["bin_offsets"], c["bin_members"], c["multiple"],
                                      c["capacity"], c["stretch"], c["width"], c["pad_value"])
            nb = len(c["bin_offsets"]) - 1
            np.testing.assert_array_equal(out.cpu().numpy().reshape(nb, -1), ref["packed"])
            np.testing.assert_array_equal(mask.cpu().numpy().reshape(nb, -1).astype(bool), ref["padding_mask"])
            np.testing.assert_array_equal(cu[:ncu].cpu().numpy(), ref["cu_flat"])
            np.testing.assert_array_equal(cup[:ncu].cpu().numpy(), ref["cu_padded_flat"])


def clear_outputs(s):
    # outputs zeroed between steps, so each check sees that step's writes
    for name, get in s._finish.items():
        for t in get():
            if isinstance(t, torch.Tensor) and t.is_cuda and t.data_ptr() not in {d.data_ptr() for d, _ in s.inputs}:
                t.zero_()
            elif isinstance(t, list):
                for d in t:
                    d[0].zero_()
    torch.cuda.synchronize(DEV)


def test_two_stream_steps_match_the_oracle(step):
    for _ in range(3):
        clear_outputs(step)
        with torch.cuda.stream(step.stream):
            step.run(two_streams=True)
        check_outputs(step)


def test_one_stream_step_matches_the_oracle(step):
    clear_outputs(step)
    with torch.cuda.stream(step.stream):
        step.run()
    check_outputs(step)


def test_torch_restatement_matches_the_oracle():
    """The bench's torch-on-GPU comparison line computes the same results."""
    import bench

    host = bench.make_inputs(1)
    calls = bench.torch_calls(host, DEV)
    for name in ("map_small", "map_stress"):
        cu, mx = calls[name]()
        ref_cu, ref_mx = oracle.from_doc_ids(host[name])
        np.testing.assert_array_equal(cu.cpu().numpy(), ref_cu)
        assert mx == ref_mx
    for name in ("thd_small", "thd_ids"):
        bt = host[name]
        cu, cup, outs, mask, mx = calls[name]()
        ref = oracle.process_input_for_thd(
            {k: bt[k] for k in ("input_ids", "labels", "position_ids", "seq_lens", "seq_lens_padded")})
        np.testing.assert_array_equal(cu.cpu().numpy(), ref["cu_seqlens"])
        np.testing.assert_array_equal(cup.cpu().numpy(), ref["cu_seqlens_padded"])
        np.testing.assert_array_equal(mask.cpu().numpy(), ref["padding_mask"])
        assert mx == ref["max_seqlen"]
        for got, key in zip(outs, ("input_ids", "labels", "position_ids")):
            np.testing.assert_array_equal(got.cpu().numpy().reshape(-1), ref[key].reshape(-1))
    c = host["squeeze"]
    out, mask, cu, cup = calls["squeeze"]()
    ref = oracle.pack_squeeze(c["src"], c["real_lens"], c["bin_offsets"], c["bin_members"], c["multiple"],
                              c["capacity"], c["stretch"], c["width"], c["pad_value"])
    np.testing.assert_array_equal(out.cpu().numpy(), ref["packed"])
    np.testing.assert_array_equal(mask.cpu().numpy(), ref["padding_mask"])
    np.testing.assert_array_equal(cu.cpu().numpy(), ref["cu_flat"])
    np.testing.assert_array_equal(cup.cpu().numpy(), ref["cu_padded_flat"])


def test_step_replayed_from_a_cuda_graph_matches_the_oracle(step):
    """The two-stream step captured once in a CUDA graph and replayed."""
    import bench

    g = bench.capture_step(step, step.stream)
    for _ in range(2):
        clear_outputs(step)
        with torch.cuda.stream(step.stream):
            g.replay()
        check_outputs(step)

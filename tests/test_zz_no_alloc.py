"""The scratch-free attention entry point (spd_attention_decode_noalloc).

It exists for callers that cannot lend device memory to the library (everything they
own is held by another allocator, or a cudaMalloc's implicit synchronisation is not
acceptable where they run); its scratch is a fixed array inside the library.  This file
is collected last on purpose, so that a run stopping at the first failure has run every
other test first.  It checks, through the C ABI, that two calls in a row (the second on
different data, after the first left its scratch behind) give what the entry point with
caller scratch gives, and that oversize shapes are refused."""
import numpy as np
import pytest
import torch

from speculative_pipeline_decoding_spd_gb300 import binding as B

pytestmark = pytest.mark.gpu

TOL = 1e-4   # the tolerance the attention parity tests use (relative to max |out|)


def _inputs(Hq, Hkv, hd, S, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(Hq, hd, generator=g).cuda()
    k = torch.randn(S, Hkv, hd, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(S, Hkv, hd, generator=g).to(torch.bfloat16).cuda()
    return q, k, v


def _with_scratch(q, k, v):
    Hq, hd = q.shape
    S, Hkv, _ = k.shape
    out = torch.empty(Hq, hd, device="cuda")
    nb = B.spd_attention_scratch_bytes(Hq, Hkv, hd, S)
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    B.spd_attention_decode(B.SPD_BF16, Hq, Hkv, hd, S, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           scratch.data_ptr(), nb, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _no_alloc(q, k, v):
    Hq, hd = q.shape
    S, Hkv, _ = k.shape
    out = torch.empty(Hq, hd, device="cuda")
    B.spd_attention_decode_noalloc(B.SPD_BF16, Hq, Hkv, hd, S, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                   out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_no_alloc_matches_caller_scratch_on_two_calls_in_a_row():
    # several chunks each, so the arrival counters and the partials are both used; the
    # second call runs on other data right after the first left its scratch behind
    cases = [(32, 8, 128, 1000, 11), (16, 2, 128, 700, 12)]
    inputs = [_inputs(Hq, Hkv, hd, S, seed) for Hq, Hkv, hd, S, seed in cases]
    refs = [_with_scratch(*x) for x in inputs]
    got = [_no_alloc(*x) for x in inputs]          # two calls in a row
    for (Hq, _, _, S, _), r, g in zip(cases, refs, got):
        err = np.max(np.abs(g - r)) / np.max(np.abs(r))
        assert err <= TOL, (Hq, S, err)


def test_no_alloc_refuses_shapes_beyond_its_buffer():
    q, k, v = _inputs(32, 8, 128, 16, 13)
    with pytest.raises(B.SPDError) as e:
        B.spd_attention_decode_noalloc(B.SPD_BF16, 32, 8, 128, 9000, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       q.data_ptr(), 0)
    assert e.value.code == B.SPD_ECAPACITY
    assert "scratch" in B.spd_ops_last_error()

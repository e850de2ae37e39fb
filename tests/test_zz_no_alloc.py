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


KV_TYPES = {B.SPD_BF16: torch.bfloat16, B.SPD_F16: torch.float16, B.SPD_F32: torch.float32}


def _inputs(Hq, Hkv, hd, S, seed, dtype=B.SPD_BF16):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(Hq, hd, generator=g).cuda()
    k = torch.randn(S, Hkv, hd, generator=g).to(KV_TYPES[dtype]).cuda()
    v = torch.randn(S, Hkv, hd, generator=g).to(KV_TYPES[dtype]).cuda()
    return q, k, v, dtype


def _with_scratch(q, k, v, dtype):
    Hq, hd = q.shape
    S, Hkv, _ = k.shape
    out = torch.empty(Hq, hd, device="cuda")
    nb = B.spd_attention_scratch_bytes(Hq, Hkv, hd, S)
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    B.spd_attention_decode(dtype, Hq, Hkv, hd, S, q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                           scratch.data_ptr(), nb, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _no_alloc(q, k, v, dtype):
    Hq, hd = q.shape
    S, Hkv, _ = k.shape
    out = torch.empty(Hq, hd, device="cuda")
    B.spd_attention_decode_noalloc(dtype, Hq, Hkv, hd, S, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                   out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_no_alloc_matches_caller_scratch_on_two_calls_in_a_row():
    # several chunks each, so the arrival counters and the partials are both used; every
    # call after the first runs on other data right after the one before left its scratch
    # behind; the K/V operand types of the call (fp32, bf16, fp16); the largest sequence that
    # fits the built-in buffer at Hq 32, hd 128 (7936 positions, 62 chunks)
    cases = [(32, 8, 128, 1000, 11, B.SPD_BF16), (16, 2, 128, 700, 12, B.SPD_BF16),
             (32, 8, 128, 900, 14, B.SPD_F32), (8, 4, 64, 333, 15, B.SPD_F16), (32, 8, 128, 7936, 16, B.SPD_F16)]
    inputs = [_inputs(Hq, Hkv, hd, S, seed, dt) for Hq, Hkv, hd, S, seed, dt in cases]
    refs = [_with_scratch(*x) for x in inputs]
    got = [_no_alloc(*x) for x in inputs]          # calls in a row
    for (Hq, _, _, S, _, _), r, g in zip(cases, refs, got):
        err = np.max(np.abs(g - r)) / np.max(np.abs(r))
        assert err <= TOL, (Hq, S, err)


def test_no_alloc_refuses_shapes_beyond_its_buffer():
    q, k, v, _ = _inputs(32, 8, 128, 16, 13)
    for S in (7937, 8064, 9000):        # 63 chunks and more need more than 1 MiB at Hq 32, hd 128
        with pytest.raises(B.SPDError) as e:
            B.spd_attention_decode_noalloc(B.SPD_BF16, 32, 8, 128, S, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                           q.data_ptr(), 0)
        assert e.value.code == B.SPD_ECAPACITY
        assert "scratch" in B.spd_ops_last_error()


def test_no_alloc_replays_inside_a_cuda_graph():
    # the first call (outside any capture) looks up the array's device address; a second call
    # captured into a graph and replayed gives what the caller-scratch entry point gives
    q, k, v, dt = _inputs(32, 8, 128, 1000, 17)
    ref = _with_scratch(q, k, v, dt)
    _no_alloc(q, k, v, dt)
    out = torch.zeros(32, 128, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        B.spd_attention_decode_noalloc(dt, 32, 8, 128, 1000, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    graph.replay()
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    assert np.max(np.abs(got - ref)) / np.max(np.abs(ref)) <= TOL

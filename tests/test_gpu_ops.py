"""GPU parity of the standalone decode attention (spd_attention_decode) against the oracle.

Shapes cover GQA groups 1..8, both head dims, fp32, bf16 and fp16 caches, and sequence
lengths of one chunk, exact chunk multiples and ragged tails over several 128-position
chunks.  The oracle gets the same rounded K and V, so every case's error is fp32
rounding only: rel 1e-4 of max |out|."""
import numpy as np
import pytest
import torch

from oracle import attend
from speculative_pipeline_decoding_spd_gb300 import binding as B

pytestmark = pytest.mark.gpu


def _case(Hq, Hkv, hd, S, dtype, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(Hq, hd, generator=g)
    k = torch.randn(S, Hkv, hd, generator=g)
    v = torch.randn(S, Hkv, hd, generator=g)
    if dtype == B.SPD_BF16:
        k, v = k.to(torch.bfloat16), v.to(torch.bfloat16)
    elif dtype == B.SPD_F16:
        k, v = k.to(torch.float16), v.to(torch.float16)
    return q, k, v


def run_attention(q, k, v, dtype):
    Hq, hd = q.shape
    S, Hkv, _ = k.shape
    dq, dk, dv = q.cuda(), k.cuda(), v.cuda()
    out = torch.empty(Hq, hd, device="cuda")
    nb = B.spd_attention_scratch_bytes(Hq, Hkv, hd, S)
    scratch = torch.empty(nb, dtype=torch.uint8, device="cuda")
    B.spd_attention_decode(dtype, Hq, Hkv, hd, S, dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), out.data_ptr(),
                           scratch.data_ptr(), nb, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    return out.cpu().numpy()


@pytest.mark.parametrize("Hq,Hkv,hd", [(4, 4, 64), (8, 4, 64), (32, 8, 128), (16, 2, 128)])
@pytest.mark.parametrize("S", [1, 77, 128, 129, 300, 1025])
@pytest.mark.parametrize("dtype", [B.SPD_F32, B.SPD_BF16, B.SPD_F16], ids=["f32", "bf16", "f16"])
def test_attention_matches_oracle(Hq, Hkv, hd, S, dtype):
    q, k, v = _case(Hq, Hkv, hd, S, dtype, seed=S * 7 + Hq)
    got = run_attention(q, k, v, dtype)
    ref = attend(q.double().numpy()[None], k.double().numpy(), v.double().numpy(), np.array([S - 1]))[0]
    err = np.max(np.abs(got - ref)) / max(1e-30, np.max(np.abs(ref)))
    assert err <= 1e-4, err


def test_attention_is_deterministic_and_rejects_bad_input():
    q, k, v = _case(32, 8, 128, 700, B.SPD_BF16, seed=3)
    a = run_attention(q, k, v, B.SPD_BF16)
    b = run_attention(q, k, v, B.SPD_BF16)
    assert np.array_equal(a, b)
    with pytest.raises(B.SPDError) as e:
        B.spd_attention_decode(B.SPD_BF16, 12, 8, 128, 10, 16, 16, 16, 16, 256, 1 << 20, 0)
    assert e.value.code == B.SPD_EINVAL
    with pytest.raises(B.SPDError) as e:
        B.spd_attention_decode(B.SPD_BF16, 32, 8, 96, 10, 16, 16, 16, 16, 256, 1 << 20, 0)
    assert e.value.code == B.SPD_EINVAL
    dq = torch.zeros(32, 128, device="cuda")
    dk = torch.zeros(10, 8, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty(32, 128, device="cuda")
    small = torch.empty(256, dtype=torch.uint8, device="cuda")
    with pytest.raises(B.SPDError) as e:
        B.spd_attention_decode(B.SPD_BF16, 32, 8, 128, 10, dq.data_ptr(), dk.data_ptr(), dk.data_ptr(),
                               out.data_ptr(), small.data_ptr(), 256, 0)
    assert e.value.code == B.SPD_ENOMEM

"""A bounded wait that runs out is reported, and the GPU context stays usable.

Every mbarrier wait in the library gives up after a bound (about 2 s of SM clock), sets an
error flag in the run state and lets the kernel finish; the host reports SPD_EDEVICE.  This
test makes one wait run out without faulting anything: the handle is created with a short
bound and a test hook under which one CTA of the first gate/up launch never loads its last
weight tile (nothing else changes; the tile's consumers time out, compute with stale shared
memory and return).  Then a fresh handle on the same context decodes exactly as a run that
never saw the hook."""
import numpy as np
import pytest
import torch

import spd_inputs as si
from gpu_common import Case, engine, materialise, run_gpu
from speculative_pipeline_decoding_spd_gb300 import binding as B

pytestmark = pytest.mark.gpu

ERR_TIMEOUT = 6
CASE = Case(si.ModelDims(L=6, d=256, Hq=4, Hkv=2, hd=64, F=512, V=2000), n=3, anchors=(0, 3, 6), Ls=2,
            prompt_len=64, max_new=24, norms="perturbed")


def test_wait_that_runs_out_reports_edevice(monkeypatch):
    reference = run_gpu(CASE)[0]
    tg, pd, prompt, m, _, _ = materialise(CASE)
    monkeypatch.setenv("SPD_TEST_WAIT_CYCLES", "2000000")      # about 1 ms
    monkeypatch.setenv("SPD_TEST_WITHHOLD_TILE", "1")
    e = engine(CASE, graph=False)
    e.prefill(torch.from_numpy(prompt).cuda())
    with pytest.raises(B.SPDError) as ex:
        e.step(1)
    assert ex.value.code == B.SPD_EDEVICE
    assert "device error flag 6" in str(ex.value)
    assert e.stats()["device_error"] == ERR_TIMEOUT
    e.close()
    monkeypatch.delenv("SPD_TEST_WAIT_CYCLES")
    monkeypatch.delenv("SPD_TEST_WITHHOLD_TILE")
    # the context is fine: a new handle decodes the same tokens as before the hook
    torch.cuda.synchronize()
    again = run_gpu(CASE)[0]
    assert again == reference
    # and generate() reports the same failure through its own path
    monkeypatch.setenv("SPD_TEST_WAIT_CYCLES", "2000000")
    monkeypatch.setenv("SPD_TEST_WITHHOLD_TILE", "1")
    e = engine(CASE, graph=True)
    with pytest.raises(B.SPDError) as ex:
        e.generate(torch.from_numpy(prompt).cuda())
    assert ex.value.code == B.SPD_EDEVICE
    e.close()
    torch.cuda.synchronize()
    assert np.isfinite(np.array(reference)).all()

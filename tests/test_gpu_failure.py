"""Failure detection without a GPU fault: a bounded wait that nothing
completes gives up after its limit, reports VCE_ERR_TIMEOUT through the status
word, and leaves the context usable. Data errors are reported, not faulted."""
import time

import numpy as np
import pytest
import torch

import vce_run as R
from vocab_embedding_cross_gb300 import device as D
from vocab_embedding_cross_gb300 import inputs as I

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    R.vce.vce_wait_selftest(5_000_000, st)          # 5 ms limit on a barrier nobody completes
    torch.cuda.synchronize()
    assert int(st.item()) == R.vce.VCE_ERR_TIMEOUT
    assert time.time() - t0 < 30
    # the context still works: a normal lookup right after
    wl = I.custom(T=64, H=64, dtype="bf16", seed=31)
    d = I.make_all(wl, ("W", "ids"))
    out = R.embed_fwd(wl, D.to_device(d["W"]), d["ids"])
    valid = (d["ids"] >= 0) & (d["ids"] < wl.V_real)
    assert np.array_equal(out["E"][valid], d["W"][d["ids"][valid]])


def test_first_error_wins():
    st = torch.full((1,), R.vce.VCE_ERR_BAD_INDEX, dtype=torch.int32, device="cuda")
    R.vce.vce_wait_selftest(1_000_000, st)
    torch.cuda.synchronize()
    assert int(st.item()) == R.vce.VCE_ERR_BAD_INDEX


def test_host_errors_enqueue_nothing():
    wl = I.custom(T=64, H=64, dtype="bf16", seed=32)
    p = R.prob(wl)
    W = torch.zeros((wl.Vp, wl.H), dtype=torch.bfloat16, device="cuda")
    E = torch.full((wl.T, wl.H), 3.0, dtype=torch.bfloat16, device="cuda")
    ids = torch.zeros(wl.T, dtype=torch.int64, device="cuda")
    bad = R.prob(wl, Vp=1000)                        # not a multiple of 64
    with pytest.raises(R.vce.VceError) as e:
        R.vce.vce_embed_fwd(bad, ids, W, E)
    assert e.value.status == R.vce.VCE_ERR_ARG
    torch.cuda.synchronize()
    assert torch.all(E == 3.0).item()                # nothing ran
    R.vce.vce_embed_fwd(p, ids, W, E)
    torch.cuda.synchronize()
    assert torch.all(E == 0.0).item()

"""A bounded wait that runs out, on the GPU, without a hang or a fault.

With the test hook SSFWD_TEST_STALL=<k> the producer warp never issues chunk k
of each CTA (so that chunk's barrier phase never completes, as if a copy were
lost) and every wait gives up after 1024 try_wait calls of at most 1 us. The
waiting warps must then leave their loops, record the code in the caller's
own error word, wait (boundedly) for the copies already in flight and
return; the context must stay usable for the next call.
"""
import ctypes
import time

import pytest
import torch

from state_space_model_03_gb300 import api, workloads

pytestmark = pytest.mark.gpu

NAMES = ("u", "delta", "A", "B", "C", "D", "z", "delta_bias")


@pytest.mark.parametrize("w,stall", [
    (workloads.Workload("stall_bf16", 1, 32, 512, 16, dtype="bf16", return_last_state=True, seed=401), 1),
    (workloads.Workload("stall_fp16", 1, 32, 512, 16, dtype="fp16", bc_dtype="fp32", seed=402), 0),
], ids=lambda v: getattr(v, "name", str(v)))
def test_a_stalled_chunk_ends_in_the_callers_error_word(w, stall, monkeypatch):
    lib = api.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    x = workloads.make_inputs(w)
    dev = {k: (None if x[k] is None else x[k].to("cuda")) for k in NAMES}
    nu = api.normalise(*(dev[k] for k in NAMES))
    ref = api.selective_scan_fn(*nu[:5], D=nu[5], z=nu[6], delta_bias=nu[7], delta_softplus=True)
    api.device_error(clear=True)
    out = torch.empty_like(nu[0])
    last = torch.empty((w.batch, w.dim, w.dstate), device="cuda") if w.return_last_state else None
    word = torch.zeros(4, dtype=torch.int32, device="cuda")
    p = api.make_params(*nu, True, out, last)
    p.error_word = word.data_ptr()
    monkeypatch.setenv("SSFWD_TEST_STALL", str(stall))
    t0 = time.time()
    assert lib.ss_fwd(ctypes.byref(p), stream) == 0  # enqueued; the failure happens on the device
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    monkeypatch.delenv("SSFWD_TEST_STALL")
    code = int(word[0])
    assert code in (1, 2, 3)              # a wait for data, a free slot or a ready slot gave up
    assert int(word[1:].abs().sum()) == 0  # only the word itself was written
    assert api.device_error() == 0         # the library's shared word was not touched
    assert elapsed < 30.0
    # the context is intact: the same call without the hook matches the earlier result
    word.zero_()
    assert lib.ss_fwd(ctypes.byref(p), stream) == 0
    torch.cuda.synchronize()
    assert int(word[0]) == 0
    assert torch.equal(out, ref)

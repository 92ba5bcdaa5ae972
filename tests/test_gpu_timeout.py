"""A bounded device-side wait that gives up (through the C ABI, on the GPU).

Every wait of a kernel for its own bulk copies has an iteration limit. sdm_set_wait_limit makes
that limit one poll, so the pipelined Phase-2 kernel's first wait gives up before its copies
land: the kernel must set SDM_ERR_TIMEOUT in the device status, let its copies in flight land
(its drain keeps the default limit) and return. Nothing faults, the context stays usable, and
the next call with the default limit is correct.
"""

import pytest
import torch

import sdm_inputs as si
import sparse_addressed_delta_gb300 as sdm
from sdm_case import TOL, compare_with_oracle, run_gpu, small_workload, to_device

pytestmark = pytest.mark.gpu


def test_wait_gives_up_reports_timeout_and_recovers():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    wl = small_workload(P=2, T=8 * 64, C=64, S=4096, D=128, W=16, R=16, dtype="bf16",
                        slots="zipf1.1", ragged=False, seed=51)
    shape = sdm.make_shape(wl.P, wl.T, wl.C, wl.S, wl.D, wl.W, wl.R, torch.bfloat16)
    assert sdm.launch_count(shape) == 3          # Phase 1, solve, the pipelined Phase 2
    inputs = si.generate(wl)
    dev = to_device(inputs, wl)
    prev = sdm.set_wait_limit(1)
    try:
        _, _, ws = run_gpu(wl, dev)
        st = sdm.device_status(ws)
    finally:
        assert sdm.set_wait_limit(prev) == 1
    assert st["code"] == -4, st                  # SDM_ERR_TIMEOUT
    r, b, ws2 = run_gpu(wl, dev)
    assert sdm.device_status(ws2)["code"] == 0
    er, eb = compare_with_oracle(wl, inputs, r, b)
    assert er <= TOL[wl.dtype] and eb <= TOL[wl.dtype], (er, eb)

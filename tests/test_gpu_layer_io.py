"""Layer I/O kernels (head split/merge, per-batch bank expand and sum) against the oracle's
array rearranges: the copies bitwise, the batch sum within the rounding of one float32 sum and
one rounding to the dtype."""

import numpy as np
import pytest
import torch

import oracle
import sparse_addressed_delta_gb300 as sdm

pytestmark = pytest.mark.gpu

DT = {"f32": torch.float32, "bf16": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    sdm.library()


def rand(shape, dtype, seed):
    x = torch.from_numpy(np.random.default_rng(seed).standard_normal(shape).astype(np.float32))
    return x.to(DT[dtype]).cuda()


def host64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,T,H,CD", [(2, 37, 4, 128), (3, 5, 8, 64), (1, 9, 3, 3), (2, 4, 5, 7)])
def test_head_split_and_merge(dtype, B, T, H, CD):
    x = rand((B, T, H * CD), dtype, B + T + H + CD)
    y = sdm.head_split(x, H)
    assert np.array_equal(host64(y), oracle.head_split(host64(x), H))
    z = sdm.head_merge(y, H)
    torch.cuda.synchronize()
    assert torch.equal(z, x)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("B,S,D", [(4, 1000, 128), (3, 17, 5), (1, 64, 32)])
def test_bank_expand_and_sum(dtype, B, S, D):
    p = rand((S, D), dtype, S + D)
    e = sdm.bank_expand(p, B)
    assert np.array_equal(host64(e), oracle.bank_expand(host64(p), B))
    x = rand((B, S, D), dtype, B * S + D)
    s = sdm.bank_sum(x)
    ref = oracle.bank_sum(host64(x))
    err = np.abs(host64(s) - ref).max() / np.abs(ref).max()
    assert err <= (1e-6 if dtype == "f32" else 8e-3), err
    # batch order, one rounding: the same inputs give the same bits
    assert torch.equal(sdm.bank_sum(x), s)


def test_layer_io_refusals():
    lib = sdm.library()
    assert lib.sdm_head_split(None, None, 1, 1, 1, 1, sdm.SDM_F32, None) == -1
    x = rand((2, 3, 4), "f32", 1)
    assert lib.sdm_bank_sum(sdm._ptr(x), sdm._ptr(x), 0, 3, 4, sdm.SDM_F32, None) == -1
    assert lib.sdm_bank_expand(sdm._ptr(x), sdm._ptr(x), 2, 3, 4, 9, None) == -1

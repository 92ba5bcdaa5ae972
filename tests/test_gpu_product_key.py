"""The product-key exact top-k on the GPU (through the C ABI) against the oracle
(oracle/product_key.py, the pages' selection rule): lin and val bit for bit, with ties, NaN,
signed zeros, one to four factors, several k and both dtypes; the backward within float32
rounding of the oracle's float64 sums."""

import numpy as np
import pytest
import torch

import sparse_addressed_delta_gb300 as sdm
from oracle import product_key as pk

pytestmark = pytest.mark.gpu


def _rows(rng, rows, factors, dtype, specials):
    x = rng.standard_normal((rows, sum(factors))).astype(np.float32)
    if specials and x.shape[1] >= 4:
        # ties inside a factor and across slot sums, NaN and signed zeros
        x[:, ::7] = np.round(x[:, ::7] * 2) / 2
        x[::3, 1] = np.nan
        x[1::4, 2] = -0.0
        x[2::4, 3] = 0.0
        x[::5, :] = np.round(x[::5, :])
    if dtype == "bf16":
        x = pk.bf16_round(x)
    return x


def _to_torch(x, dtype):
    t = torch.from_numpy(x)
    return (t.bfloat16() if dtype == "bf16" else t).cuda()


CASES = [((64,), 7), ((64,), 256), ((300,), 256), ((32, 48), 1), ((32, 48), 64),
         ((16, 16), 256), ((40, 7), 256), ((16, 20, 24), 64), ((8, 9, 10, 11), 256),
         ((4096, 3), 256), ((5, 5, 5, 5), 17), ((1, 1), 5)]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("factors,k", CASES)
def test_topk_bitwise(factors, k, dtype):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    rng = np.random.default_rng(sum(factors) * 31 + k)
    x = _rows(rng, 37, factors, dtype, specials=True)
    val_ref, lin_ref = pk.product_key_topk(x, factors, k, dtype)
    val, lin = sdm.product_key_topk(_to_torch(x, dtype), factors, k)
    torch.cuda.synchronize()
    assert np.array_equal(lin.cpu().numpy(), lin_ref)
    got = val.float().cpu().numpy()
    nan = np.isnan(val_ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), val_ref[~nan].astype(np.float32).view(np.uint32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_topk_backward(dtype):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    factors, k = (16, 20, 24), 128
    rng = np.random.default_rng(7)
    x = _rows(rng, 9, factors, dtype, specials=False)
    _, lin = sdm.product_key_topk(_to_torch(x, dtype), factors, k)
    g = rng.standard_normal(lin.shape).astype(np.float32)
    if dtype == "bf16":
        g = pk.bf16_round(g)
    graw = sdm.product_key_topk_backward(lin, _to_torch(g, dtype), factors, k)
    torch.cuda.synchronize()
    ref = pk.product_key_topk_backward(lin.cpu().numpy(), g.astype(np.float64), factors)
    err = np.abs(graw.cpu().numpy() - ref).max() / np.abs(ref).max()
    assert err <= 1e-6, err

"""lmoe_permute_noalloc: the permute for callers that cannot provide a
workspace or allow any device allocation (plugin code inside another
runtime's memory pool, serving loops with memory fixed at start-up).

It is checked through the C ABI against lmoe_permute on the same inputs, on
two calls in a row (the shared fixed array keeps the previous call's
contents, so the second call must not depend on them).  This file is
collected last so that a failure here leaves every other test already run.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    score = rng.standard_normal((T, E)) - 2.0 * np.log1p(np.arange(E))[None, :] * (seed % 2)
    return np.argsort(-score, 1, kind="stable")[:, :k].astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(64, 896, 16), (3000, 896, 16), (32768, 896, 16), (700, 2048, 8)])
def test_permute_noalloc_matches_permute_twice(cuda_lib, T, E, k):
    """Both entry points against each other and against the oracle's counting
    sort (the 32768-token case is the block workload's 524,288 pairs)."""
    lmoe = cuda_lib
    for call in range(2):  # two calls in a row, different inputs
        idx_h = _routing(T, E, k, seed=T + call)
        idx = torch.from_numpy(idx_h).to(DEV)
        ref = lmoe.permute(idx, E)[:4]
        got = lmoe.permute_noalloc(idx, E)
        torch.cuda.synchronize()
        for a, b in zip(ref, got[:4]):
            assert torch.equal(a, b)
        assert int(got[4].item()) == lmoe.OK
        for a, b in zip(oracle.permute(idx_h, E), got[:4]):
            np.testing.assert_array_equal(b.cpu().numpy(), a)


def test_permute_noalloc_into_preallocated_outputs_twice(cuda_lib):
    """With every output preallocated by the caller the call allocates
    nothing; two calls in a row into the same tensors, the second on
    different routing, each equal to the oracle."""
    lmoe = cuda_lib
    T, E, k = 1024, 896, 16
    out = (torch.empty(E, dtype=torch.int32, device=DEV), torch.empty(E + 1, dtype=torch.int32, device=DEV),
           torch.empty(T * k, dtype=torch.int32, device=DEV), torch.empty(T * k, dtype=torch.int32, device=DEV),
           torch.empty(1, dtype=torch.int32, device=DEV))
    for call in range(2):
        idx_h = _routing(T, E, k, seed=11 + call)
        got = lmoe.permute_noalloc(torch.from_numpy(idx_h).to(DEV), E, out=out)
        torch.cuda.synchronize()
        assert all(a is b for a, b in zip(got, out))
        assert int(out[4].item()) == lmoe.OK
        for a, b in zip(oracle.permute(idx_h, E), out[:4]):
            np.testing.assert_array_equal(b.cpu().numpy(), a)
    bad = (out[0][:-1],) + out[1:]
    with pytest.raises(ValueError):
        lmoe.permute_noalloc(torch.from_numpy(_routing(T, E, k, seed=3)).to(DEV), E, out=bad)


def test_permute_noalloc_rejects_oversize_and_flags_bad_ids(cuda_lib):
    lmoe = cuda_lib
    T = lmoe.PERMUTE_NOALLOC_MAX_PAIRS // 16 + 1
    big = torch.zeros((T, 16), dtype=torch.int32, device=DEV)
    with pytest.raises(lmoe.LmoeError) as ei:
        lmoe.permute_noalloc(big, 896)
    assert ei.value.code == lmoe.ERR_INVALID_ARG
    idx = torch.from_numpy(np.tile(np.arange(16, dtype=np.int32), (10, 1))).to(DEV)
    idx[3, 5] = 900
    got = lmoe.permute_noalloc(idx, 896)
    torch.cuda.synchronize()
    assert int(got[4].item()) == lmoe.ERR_DEVICE_CHECK
    ok = lmoe.permute_noalloc(idx.clamp(max=895), 896)  # the status word is cleared per call
    torch.cuda.synchronize()
    assert int(ok[4].item()) == lmoe.OK

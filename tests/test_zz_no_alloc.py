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

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _routing(T, E, k, seed):
    rng = np.random.default_rng(seed)
    score = rng.standard_normal((T, E)) - 2.0 * np.log1p(np.arange(E))[None, :] * (seed % 2)
    return np.argsort(-score, 1, kind="stable")[:, :k].astype(np.int32)


@pytest.mark.parametrize("T,E,k", [(64, 896, 16), (3000, 896, 16), (32768, 896, 16), (700, 2048, 8)])
def test_permute_noalloc_matches_permute_twice(cuda_lib, T, E, k):
    lmoe = cuda_lib
    for call in range(2):  # two calls in a row, different inputs
        idx = torch.from_numpy(_routing(T, E, k, seed=T + call)).to(DEV)
        ref = lmoe.permute(idx, E)[:4]
        got = lmoe.permute_noalloc(idx, E)
        torch.cuda.synchronize()
        for a, b in zip(ref, got[:4]):
            assert torch.equal(a, b)
        assert int(got[4].item()) == lmoe.OK


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

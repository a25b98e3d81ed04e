"""The workspace-free permutation entry point (moe_permute_static_ws) against
the regular one, through the C ABI.

moe_permute_static_ws keeps its scratch in a fixed device array owned by the
library, for callers that cannot allocate device memory where they call it.
This file is collected last so that a failure here does not hide the other
tests' results; it passes on its own in a fresh process as well.
"""
import numpy as np
import pytest
import torch

from nvfp4_block_scaled_05_gb300 import binding as B

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ids(T, k, E, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randint(0, E, (T, k), dtype=torch.int32, generator=g).to(DEV)


def test_static_scratch_permutation_matches_workspace_version_twice():
    # two calls in a row with different inputs: the shared array keeps the
    # first call's contents, which must not leak into the second result
    for T, k, E, seed in [(5000, 8, 256, 1), (777, 6, 1000, 2), (16384, 8, 256, 3)]:
        ids = _ids(T, k, E, seed)
        ref = [t.cpu() for t in B.moe_permute(ids, E)]
        got = [t.cpu() for t in B.moe_permute_static_ws(ids, E)]
        torch.cuda.synchronize()
        for a, b in zip(ref, got):
            assert torch.equal(a, b), (T, k, E)


def test_static_scratch_rejects_oversized_requests():
    lib = B.lib()
    # ceil(T*k/1024) * E > 262144 entries: rejected before any launch
    st = lib.moe_permute_static_ws(None, 300000, 8, 1024, None, None, None, None)
    assert st == -3
    # the library still works afterwards
    ids = _ids(64, 2, 8, 4)
    assert all(torch.equal(a.cpu(), b.cpu())
               for a, b in zip(B.moe_permute(ids, 8), B.moe_permute_static_ws(ids, 8)))

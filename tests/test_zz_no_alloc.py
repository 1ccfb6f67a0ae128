"""moe_permute_noalloc: the permutation for callers that cannot allocate.

Some callers cannot call cudaMalloc or pass a workspace (a plugin whose host
framework owns all device memory, a serving loop that must not allocate after
start-up).  moe_permute_noalloc keeps its scratch in a fixed array inside the
library instead.  These tests call it through the C ABI twice in a row, on
different inputs that need the multi-chunk scratch, and require the same
bits as moe_permute with a caller workspace; they also check that a request
larger than the fixed scratch is refused with a message.  This file is
collected last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

import bit_expert_ffn_gb300 as m

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ids(T, k, E, seed):
    rng = np.random.default_rng(seed)
    return np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)


def _run(fn, ids, T, k, E, **kw):
    off = torch.full((E + 1,), -7, dtype=torch.int32, device=DEV)
    perm = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((T * k,), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn(torch.from_numpy(ids).to(DEV), T, k, E, off, perm, inv, dev_status=st, **kw)
    assert m.moe_check_status(st) == 0
    return off.cpu().numpy(), perm.cpu().numpy(), inv.cpu().numpy()


def test_noalloc_permute_matches_workspace_permute_on_two_calls(moe):
    for T, k, E, seed in ((6000, 10, 512, 1), (4100, 8, 1024, 2)):  # 30 and 17 chunks of scratch
        ids = _ids(T, k, E, seed)
        nb = m.moe_permute_workspace_size(T, k, E)
        ws = torch.empty(nb, dtype=torch.uint8, device=DEV)
        want = _run(m.moe_permute, ids, T, k, E, ws=ws, ws_bytes=nb)
        got = _run(m.moe_permute_noalloc, ids, T, k, E)
        for a, b in zip(got, want):
            assert np.array_equal(a, b)


def test_noalloc_permute_refuses_more_than_its_scratch(moe):
    T, k, E = 7000, 10, 1024  # 35 chunks x 1024 experts > 32,768 counters
    ids = torch.zeros(T, k, dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    with pytest.raises(m.MoeError) as e:
        m.moe_permute_noalloc(ids, T, k, E, off, perm, perm)
    assert e.value.status == m.MOE_ERR_INVALID_ARG
    assert "32768" in str(e.value)

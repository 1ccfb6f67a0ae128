"""moe_permute_noalloc: the permutation for callers that cannot allocate.

Some callers cannot call cudaMalloc or pass a workspace (a plugin whose host
framework owns all device memory, a serving loop that must not allocate after
start-up).  moe_permute_noalloc keeps its scratch in a fixed array inside the
library instead.  These tests call it through the C ABI and require the same
bits (outputs and status word) as moe_permute with a caller workspace: twice
in a row on different inputs that need the multi-chunk scratch, then a
single-chunk call right after a multi-chunk one (the shared array then holds
the earlier call's counters), an empty call, and a call with an id equal to
E (MOE_ERR_BOUNDS, that pair's inv_perm entry -1).  A request larger than the
fixed scratch is refused with a message.  This file is collected last so that
a run stopping at the first failure has already run every other test.
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
    perm = torch.full((max(T * k, 1),), -7, dtype=torch.int32, device=DEV)
    inv = torch.full((max(T * k, 1),), -7, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    fn(torch.from_numpy(ids).to(DEV), T, k, E, off, perm, inv, dev_status=st, **kw)
    status = m.moe_check_status(st)
    return status, off.cpu().numpy(), perm.cpu().numpy()[:T * k], inv.cpu().numpy()[:T * k]


def _both(ids, T, k, E):
    nb = m.moe_permute_workspace_size(T, k, E)
    ws = torch.empty(max(nb, 1), dtype=torch.uint8, device=DEV)
    want = _run(m.moe_permute, ids, T, k, E, ws=ws, ws_bytes=nb)
    got = _run(m.moe_permute_noalloc, ids, T, k, E)
    assert got[0] == want[0]
    for a, b in zip(got[1:], want[1:]):
        assert np.array_equal(a, b)
    return got


def test_noalloc_permute_matches_workspace_permute_on_two_calls(moe):
    for T, k, E, seed in ((6000, 10, 512, 1), (4100, 8, 1024, 2)):  # 30 and 17 chunks of scratch
        st, *_ = _both(_ids(T, k, E, seed), T, k, E)
        assert st == 0


def test_noalloc_permute_single_chunk_after_multi_chunk(moe):
    _both(_ids(6000, 10, 512, 3), 6000, 10, 512)
    st, off, perm, inv = _both(_ids(200, 10, 512, 4), 200, 10, 512)  # 2,000 pairs: one chunk
    assert st == 0 and off[-1] == 2000


def test_noalloc_permute_empty_and_bad_id(moe):
    st, off, _, _ = _both(np.zeros((0, 4), np.int32), 0, 4, 64)
    assert st == 0 and np.all(off == 0)
    ids = _ids(3000, 4, 64, 5)
    ids[17, 2] = 64  # == E
    ids[2999, 0] = 64
    st, off, perm, inv = _both(ids, 3000, 4, 64)
    assert st == m.MOE_ERR_BOUNDS
    assert off[-1] == 3000 * 4 - 2
    assert inv[17 * 4 + 2] == -1 and inv[2999 * 4] == -1


def test_noalloc_permute_refuses_more_than_its_scratch(moe):
    T, k, E = 7000, 10, 1024  # 35 chunks x 1024 experts > 32,768 counters
    ids = torch.zeros(T, k, dtype=torch.int32, device=DEV)
    off = torch.empty(E + 1, dtype=torch.int32, device=DEV)
    perm = torch.empty(T * k, dtype=torch.int32, device=DEV)
    with pytest.raises(m.MoeError) as e:
        m.moe_permute_noalloc(ids, T, k, E, off, perm, perm)
    assert e.value.status == m.MOE_ERR_INVALID_ARG
    assert "32768" in str(e.value)

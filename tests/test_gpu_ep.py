"""Expert parallelism through the library on one GPU: the shards of a layer
(experts split over G ranks by moe_shard_ids + moe_permute + moe_expert_forward
on each shard's own arena, the shared expert on rank 0) run one after another,
and their summed outputs equal the whole layer (the sum the ranks' all-reduce
forms) and the oracle.  Also: MOE_ID_NOT_LOCAL pairs are left out without an
error, while other out-of-range ids still report MOE_ERR_BOUNDS."""
import numpy as np
import pytest
import torch

import bit_expert_ffn_gb300 as m
import oracle
from bit_expert_ffn_gb300 import synth
from bit_expert_ffn_gb300.model import LayerShape, MoeLayer, ShardedMoeLayer, StepBuffers, Workspace
from helpers import host_layer, rel_l2

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_shard_ids_and_not_local_pairs(moe):
    rng = np.random.default_rng(1)
    ids = np.stack([rng.permutation(40)[:6] for _ in range(50)]).astype(np.int32)
    local = torch.empty(50, 6, dtype=torch.int32, device=DEV)
    m.moe_shard_ids(torch.from_numpy(ids).to(DEV), 300, 10, 12, local)
    want = np.where((ids >= 10) & (ids < 22), ids - 10, -1)
    got = local.cpu().numpy()
    assert np.array_equal(got, want)
    off = torch.empty(13, dtype=torch.int32, device=DEV)
    perm = torch.empty(300, dtype=torch.int32, device=DEV)
    inv = torch.empty(300, dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    m.moe_permute(local, 50, 6, 12, off, perm, inv, None, 0, st)
    assert m.moe_check_status(st) == 0
    keep = want >= 0
    oo, op, _ = oracle.permute(np.where(keep, want, 0)[keep].reshape(-1, 1), 12)
    assert np.array_equal(off.cpu().numpy(), oo)
    flat = np.nonzero(keep.ravel())[0]
    assert np.array_equal(perm.cpu().numpy()[:keep.sum()], flat[op])
    assert np.all(inv.cpu().numpy()[~keep.ravel()] == -1)


@pytest.mark.parametrize("world", [2, 3, 4])
@pytest.mark.parametrize("T,path", [(4, m.MOE_PATH_DECODE), (300, m.MOE_PATH_PREFILL)])
def test_shards_sum_to_the_layer(moe, world, T, path):
    s = LayerShape(H=256, I=128, E=16, k=4, Is=128, bits=2)
    seed, layer = 7, 3
    full = MoeLayer(s, DEV)
    full.fill_device(seed, layer, zipf_s=1.1)
    shards = [ShardedMoeLayer(s, r, world, DEV) for r in range(world)]
    for sh in shards:
        sh.fill_device(seed, layer, zipf_s=1.1)
    x = synth.activations(seed, T, s.H) if T > 4 else synth.verify_window(seed, T, s.H)
    xd = torch.from_numpy(x.view(np.int16)).to(DEV)
    ref = torch.zeros(T, s.H, dtype=torch.float32, device=DEV)
    bufs = StepBuffers(T, s.E, s.k, DEV)
    full.forward(xd, T, ref, Workspace(DEV), bufs, accumulate=False, path=path)
    ids, w = bufs.ids.cpu().numpy(), bufs.w.cpu().numpy()
    parts = []
    for sh in shards:
        out = torch.zeros(T, s.H, dtype=torch.float32, device=DEV)
        b = StepBuffers(T, s.E, s.k, DEV)
        sh.forward(xd, T, out, Workspace(DEV), b, path=path)
        assert m.moe_check_status(sh.status) == 0, m.moe_last_error()
        assert np.array_equal(b.ids.cpu().numpy(), ids)  # the replicated router agrees
        parts.append(out)
    total = torch.stack(parts).sum(0).cpu().numpy()
    assert rel_l2(total, ref.cpu().numpy()) <= 1e-6
    arena, _, _, shared = host_layer(seed=seed, layer=layer, bits=2, H=s.H, I=s.I, E=s.E, Is=s.Is, zipf=1.1)
    want = oracle.moe_layer(2, x, ids, w.astype(np.float64), *arena, shared=shared)
    tol = 2e-5 if path == m.MOE_PATH_DECODE else 1e-3
    assert rel_l2(total, want) <= tol

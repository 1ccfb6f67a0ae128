"""Resident MoE layers on one GPU, driven through the C ABI.

Weights are drawn with the seeded generator (host numpy for small shapes,
the device generator of ``libmoe_synth.so`` for full-size arenas), packed by
``moe_pack_experts`` and kept in HBM.  :meth:`MoeLayer.forward` runs one
layer as the sequence of library calls

    router_topk -> permute -> shared_expert -> expert_forward

writing ``out = residual + S(x) + sum_j w_j FFN_j(x)`` in fp32.  Nothing here
computes any part of the layer itself.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np
import torch

from . import (MOE_F32, MOE_PATH_AUTO, RMS_EPS, load, make_arena, moe_expert_forward, moe_expert_forward_workspace_size,
               moe_f32_to_bf16, moe_pack_experts, moe_permute, moe_permute_workspace_size, moe_rms_norm_bf16,
               moe_router_topk, moe_router_workspace_size, moe_shard_ids, moe_shared_expert,
               moe_shared_expert_workspace_size, synth, synth_lib)


def _u16(a: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev)


def device_codes(key: int, n: int, bits: int, out: torch.Tensor, start: int = 0):
    r = synth_lib().moe_synth_codes(key, start, n, bits, out.data_ptr(),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if r != 0:
        raise RuntimeError(f"moe_synth_codes failed ({r})")


def device_normal(key: int, n: int, sigma: float, kind: int, out: torch.Tensor, start: int = 0):
    """kind 0: fp32 N(0, sigma); 1: bf16 N(0, sigma); 2: fp16 |N(0, sigma)|."""
    r = synth_lib().moe_synth_normal(key, start, n, float(synth.IH_SCALE), float(np.float32(sigma)), kind,
                                     out.data_ptr(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    if r != 0:
        raise RuntimeError(f"moe_synth_normal failed ({r})")


def draw_expert_parts(seed, layer, experts, bits, H, I, dev="cuda"):
    """Logical codes and fp16 scales of the given experts from the seeded
    generator's device implementation (the streams of synth.expert_codes and
    synth.expert_scales, to which it is tested equal), copied to the host.
    Returns six numpy arrays [n][...]: gate codes, gate scales, up codes, up
    scales, down codes, down scales (the order oracle.moe_layer takes)."""
    n = len(experts)
    gu = torch.empty(n, 2 * I * H, dtype=torch.uint8, device=dev)
    d = torch.empty(n, H * I, dtype=torch.uint8, device=dev)
    gus = torch.empty(n, 2 * I * (H // 32), dtype=torch.int16, device=dev)
    ds = torch.empty(n, H * (I // 32), dtype=torch.int16, device=dev)
    for j, e in enumerate(experts):
        e = int(e)
        device_codes(synth.stream_key(seed, synth.TAG_GU_CODES, layer, e), 2 * I * H, bits, gu[j])
        device_codes(synth.stream_key(seed, synth.TAG_D_CODES, layer, e), H * I, bits, d[j])
        device_normal(synth.stream_key(seed, synth.TAG_GU_SCALES, layer, e), 2 * I * (H // 32), 0.02, 2, gus[j])
        device_normal(synth.stream_key(seed, synth.TAG_D_SCALES, layer, e), H * (I // 32), 0.02, 2, ds[j])
    gu = gu.cpu().numpy().reshape(n, 2, I, H)
    gus = gus.cpu().numpy().view(np.uint16).reshape(n, 2, I, H // 32)
    d = d.cpu().numpy().reshape(n, H, I)
    ds = ds.cpu().numpy().view(np.uint16).reshape(n, H, I // 32)
    return [np.ascontiguousarray(a) for a in (gu[:, 0], gus[:, 0], gu[:, 1], gus[:, 1], d, ds)]


@dataclass
class LayerShape:
    H: int = 2048
    I: int = 768
    E: int = 512
    k: int = 10
    Is: int = 768
    bits: int = 2


class Workspace:
    """One growing device byte buffer shared by the calls of a layer."""

    def __init__(self, dev):
        self.dev = dev
        self.buf = torch.empty(0, dtype=torch.uint8, device=dev)

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf.numel() < nbytes:
            self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.dev)
        return self.buf


class MoeLayer:
    """One routed-expert layer resident on the device."""

    def __init__(self, shape: LayerShape, dev="cuda"):
        load()
        self.s = shape
        self.dev = torch.device(dev)
        H, I, E, bits = shape.H, shape.I, shape.E, shape.bits
        cgu, sgu = _pk(bits, 2 * I, H)
        cd, sd = _pk(bits, H, I)
        self.gu_codes = torch.empty(E * cgu, dtype=torch.uint8, device=self.dev)
        self.gu_scales = torch.empty(E * sgu // 2, dtype=torch.int16, device=self.dev)
        self.d_codes = torch.empty(E * cd, dtype=torch.uint8, device=self.dev)
        self.d_scales = torch.empty(E * sd // 2, dtype=torch.int16, device=self.dev)
        self.router_w = torch.empty(E, H, dtype=torch.float32, device=self.dev)
        self.router_b = torch.zeros(E, dtype=torch.float32, device=self.dev)
        self.shared = None
        self.status = torch.zeros(1, dtype=torch.int32, device=self.dev)
        self.arena = make_arena(bits, H, I, E, self.gu_codes, self.gu_scales, self.d_codes, self.d_scales)

    # -- filling --------------------------------------------------------
    def load_host(self, gate, gate_s, up, up_s, down, down_s, router_w, router_b=None, shared=None):
        """Logical codes [E][I][H] / [E][H][I] and fp16-bit scales from the host; packed on the device."""
        s = self.s
        gu = np.concatenate([gate, up], axis=1)  # [E][2I][H]
        gus = np.concatenate([gate_s, up_s], axis=1)
        self._pack(gu, gus, self.gu_codes, self.gu_scales, 2 * s.I, s.H)
        self._pack(down, down_s, self.d_codes, self.d_scales, s.H, s.I)
        self.router_w.copy_(torch.from_numpy(np.ascontiguousarray(router_w, np.float32)))
        if router_b is not None:
            self.router_b.copy_(torch.from_numpy(np.ascontiguousarray(router_b, np.float32)))
        if shared is not None:
            self.shared = tuple(_u16(a, self.dev) for a in shared)

    def _pack(self, codes, scales, pc, ps, rows, cols):
        E = self.s.E
        c = torch.from_numpy(np.ascontiguousarray(codes, np.uint8).reshape(-1)).to(self.dev)
        sc = _u16(np.asarray(scales, np.uint16).reshape(-1), self.dev)
        moe_pack_experts(self.s.bits, E, rows, cols, c, sc, pc, ps, self.status)

    def fill_device(self, seed: int, layer: int, zipf_s: float = 0.0, chunk_experts: int = 64, expert_base: int = 0):
        """Draw every tensor of the layer on the device with the seeded generator and pack it.  With
        expert_base > 0 the arena holds experts expert_base .. expert_base + E - 1 of the layer (a shard)."""
        s = self.s
        H, I, E, bits = s.H, s.I, s.E, s.bits
        for mat, (rows, cols, tag_c, tag_s, pc, ps) in enumerate((
                (2 * I, H, synth.TAG_GU_CODES, synth.TAG_GU_SCALES, self.gu_codes, self.gu_scales),
                (H, I, synth.TAG_D_CODES, synth.TAG_D_SCALES, self.d_codes, self.d_scales))):
            cb, sb = _pk(bits, rows, cols)
            per = rows * cols
            nsc = rows * cols // 32
            tmp_c = torch.empty(min(E, chunk_experts) * per, dtype=torch.uint8, device=self.dev)
            tmp_s = torch.empty(min(E, chunk_experts) * nsc, dtype=torch.int16, device=self.dev)
            for e0 in range(0, E, chunk_experts):
                ne = min(chunk_experts, E - e0)
                for j in range(ne):
                    e = expert_base + e0 + j
                    device_codes(synth.stream_key(seed, tag_c, layer, e), per, bits, tmp_c[j * per:(j + 1) * per])
                    device_normal(synth.stream_key(seed, tag_s, layer, e), nsc, 0.02, 2, tmp_s[j * nsc:(j + 1) * nsc])
                moe_pack_experts(bits, ne, rows, cols, tmp_c, tmp_s, pc[e0 * cb:(e0 + ne) * cb],
                                 ps[e0 * sb // 2:(e0 + ne) * sb // 2], self.status)
            del tmp_c, tmp_s
        device_normal(synth.stream_key(seed, synth.TAG_ROUTER, layer), E * H, 0.02, 0, self.router_w)
        self.router_b.copy_(torch.from_numpy(synth.zipf_bias(seed, layer, E, zipf_s)))
        sh = []
        for tag, n in ((synth.TAG_SHARED_G, s.Is * H), (synth.TAG_SHARED_U, s.Is * H), (synth.TAG_SHARED_D, H * s.Is)):
            t = torch.empty(n, dtype=torch.int16, device=self.dev)
            device_normal(synth.stream_key(seed, tag, layer), n, 0.02, 1, t)
            sh.append(t)
        self.shared = tuple(sh)

    def weights(self):
        """This layer as a moe_layer_weights descriptor for moe_decode_forward."""
        from . import moe_layer_weights

        sh = self.shared
        return moe_layer_weights(self.arena, self.router_w.data_ptr(), self.router_b.data_ptr(),
                                 sh[0].data_ptr() if sh else None, sh[1].data_ptr() if sh else None,
                                 sh[2].data_ptr() if sh else None, self.s.Is if sh else 0)

    # -- running --------------------------------------------------------
    def forward(self, x_bf16, T, out_f32, ws: Workspace, bufs: "StepBuffers", accumulate=True, path=MOE_PATH_AUTO,
                with_shared=True):
        """out_f32 (+)= S(x) + routed(x), through the library calls only."""
        s = self.s
        rws = moe_router_workspace_size(T, s.H, s.E, True)
        pws = moe_permute_workspace_size(T, s.k, s.E)
        ews = moe_expert_forward_workspace_size(self.arena, T, s.k, path)
        sws = moe_shared_expert_workspace_size(s.H, s.Is, T) if with_shared and self.shared is not None else 0
        need = max(rws, pws, ews, sws)
        buf = ws.get(need)
        moe_router_topk(x_bf16, T, s.H, self.router_w, self.router_b, s.E, s.k, bufs.logits, bufs.ids, bufs.w,
                        buf if rws else None, rws, dev_status=self.status)
        moe_permute(bufs.ids, T, s.k, s.E, bufs.offsets, bufs.perm, bufs.inv, buf if pws else None, pws,
                    dev_status=self.status)
        acc = accumulate
        if with_shared and self.shared is not None:
            moe_shared_expert(*self.shared, s.H, s.Is, x_bf16, T, out_f32, MOE_F32, acc, buf, sws,
                              dev_status=self.status)
            acc = True
        moe_expert_forward(self.arena, x_bf16, T, bufs.ids, bufs.w, s.k, bufs.offsets, bufs.perm, bufs.inv, out_f32,
                           MOE_F32, acc, path, buf, ews, dev_status=self.status)


class StepBuffers:
    """Routing buffers for up to T tokens."""

    def __init__(self, T, E, k, dev="cuda"):
        d = torch.device(dev)
        self.logits = torch.empty(max(T, 1), E, dtype=torch.float32, device=d)
        self.ids = torch.empty(max(T, 1), k, dtype=torch.int32, device=d)
        self.w = torch.empty(max(T, 1), k, dtype=torch.float32, device=d)
        self.offsets = torch.empty(E + 1, dtype=torch.int32, device=d)
        self.local_ids = torch.empty(max(T, 1), k, dtype=torch.int32, device=d)  # a shard's ids (expert parallelism)
        self.perm = torch.empty(max(T * k, 1), dtype=torch.int32, device=d)
        self.inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=d)


def residual_step(layers, x_res, x_bf16, T, ws, bufs, path=MOE_PATH_AUTO, rms_eps=RMS_EPS):
    """x_res <- x_res + MoE_l(bf16(x_res / rms(x_res))) for every layer, in place (fp32 residual stream)."""
    for L in layers:
        if rms_eps is None:
            moe_f32_to_bf16(x_res, x_bf16, x_res.numel())
        else:
            moe_rms_norm_bf16(x_res, x_bf16, T, L.s.H, rms_eps)
        L.forward(x_bf16, T, x_res, ws, bufs, accumulate=True, path=path)


def _pk(bits, rows, cols):
    from . import moe_packed_size

    return moe_packed_size(bits, rows, cols)


# ---------------------------------------------------------------- expert parallelism

def expert_shards(E: int, world: int):
    """Contiguous, balanced expert ranges [e0, e1) of a layer for `world` shards (the first E % world
    shards hold one expert more); together they cover [0, E) once."""
    if world < 1 or world > E:
        raise ValueError(f"cannot split {E} experts over {world} shards")
    base, extra = divmod(E, world)
    out, e0 = [], 0
    for r in range(world):
        n = base + (1 if r < extra else 0)
        out.append((e0, e0 + n))
        e0 += n
    return out


def ep_all_reduce(out: torch.Tensor, group=None):
    """Sum a shard's partial layer output over the ranks of `group` in place (NCCL on GPUs, gloo on CPU)."""
    import torch.distributed as dist

    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(out, op=dist.ReduceOp.SUM, group=group)
    return out


class ShardedMoeLayer:
    """One layer's experts [e0, e1) on this rank (expert parallelism), the router replicated on every rank and
    the shared expert on rank 0 only.  forward() adds this rank's part of the layer to `out`; after
    ep_all_reduce over the ranks every rank holds the whole layer.  Activations are replicated (every rank
    has every token), so no dispatch of token rows is needed: each rank computes the pairs routed to its
    experts and the reduction combines them."""

    def __init__(self, shape: LayerShape, rank: int, world: int, dev="cuda"):
        self.s = shape
        self.rank, self.world = rank, world
        self.e0, self.e1 = expert_shards(shape.E, world)[rank]
        local = LayerShape(H=shape.H, I=shape.I, E=self.e1 - self.e0, k=shape.k, Is=shape.Is, bits=shape.bits)
        self.local = MoeLayer(local, dev)
        self.dev = self.local.dev
        self.router_w = torch.empty(shape.E, shape.H, dtype=torch.float32, device=self.dev)
        self.router_b = torch.zeros(shape.E, dtype=torch.float32, device=self.dev)
        self.status = self.local.status

    def fill_device(self, seed: int, layer: int, zipf_s: float = 0.0):
        s = self.s
        self.local.fill_device(seed, layer, zipf_s, expert_base=self.e0)
        device_normal(synth.stream_key(seed, synth.TAG_ROUTER, layer), s.E * s.H, 0.02, 0, self.router_w)
        self.router_b.copy_(torch.from_numpy(synth.zipf_bias(seed, layer, s.E, zipf_s)))
        if self.rank != 0:
            self.local.shared = None

    def forward(self, x_bf16, T, out_f32, ws: Workspace, bufs: "StepBuffers", path=MOE_PATH_AUTO):
        """out_f32 += (rank 0: S(x)) + sum over this rank's pairs of w_j FFN_j(x), through library calls only."""
        s, L = self.s, self.local
        El = self.e1 - self.e0
        rws = moe_router_workspace_size(T, s.H, s.E, True)
        pws = moe_permute_workspace_size(T, s.k, El)
        ews = moe_expert_forward_workspace_size(L.arena, T, s.k, path)
        sws = moe_shared_expert_workspace_size(s.H, s.Is, T) if L.shared is not None else 0
        buf = ws.get(max(rws, pws, ews, sws))
        moe_router_topk(x_bf16, T, s.H, self.router_w, self.router_b, s.E, s.k, bufs.logits, bufs.ids, bufs.w,
                        buf if rws else None, rws, dev_status=self.status)
        moe_shard_ids(bufs.ids, T * s.k, self.e0, El, bufs.local_ids)
        moe_permute(bufs.local_ids, T, s.k, El, bufs.offsets, bufs.perm, bufs.inv, buf if pws else None, pws,
                    dev_status=self.status)
        if L.shared is not None:
            moe_shared_expert(*L.shared, s.H, s.Is, x_bf16, T, out_f32, MOE_F32, True, buf, sws,
                              dev_status=self.status)
        moe_expert_forward(L.arena, x_bf16, T, bufs.local_ids, bufs.w, s.k, bufs.offsets, bufs.perm, bufs.inv,
                           out_f32, MOE_F32, True, path, buf, ews, dev_status=self.status)

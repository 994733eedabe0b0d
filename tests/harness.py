"""Shared set-up for the GPU parity tests: the same seeded inputs go to the
library (through its C ABI) and to the oracle; each side computes slots,
appends, quantisation and attention on its own."""

import math

import numpy as np
import torch

import synth
from oracle import attention as oatt
from oracle import cache as ocache
from oracle import numerics
from synth import workloads

TOL = {"f32": 1e-5, "f16": 1e-2, "bf16": 1e-2, "fp8_e4m3": 3e-2}
POISON = 0xFF   # NaN in every float type and in E4M3: unused slots must never be read


def to_torch(arr, dtype, device):
    """Host storage array (float32 / float16 / bf16 bits / e4m3 codes) -> torch tensor."""
    if dtype == "bf16":
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).to(device)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(device)


def to_numpy_storage(t, dtype):
    a = t.detach().cpu()
    if dtype == "bf16":
        return a.view(torch.int16).numpy().view(np.uint16)
    return a.numpy()


class Case:
    """A decode problem with explicit shapes, drawn from a seed."""

    def __init__(self, *, batch, hq, hkv, d, bs, kv_dtype, q_dtype, ctx, seed, spare_blocks=3,
                 partition=0, src_dtype=None):
        self.batch, self.hq, self.hkv, self.d, self.bs = batch, hq, hkv, d, bs
        self.kv_dtype, self.q_dtype = kv_dtype, q_dtype
        self.ctx = np.asarray(ctx, dtype=np.int32)
        self.partition = partition
        self.src_dtype = src_dtype or ("f32" if kv_dtype == "fp8_e4m3" else kv_dtype)
        nblk = [-(-int(c) // bs) for c in self.ctx]
        self.max_blocks = max(1, max(nblk))
        self.num_blocks = sum(nblk) + spare_blocks
        perm = synth.permutation(seed, 100, self.num_blocks)
        self.tables = np.zeros((batch, self.max_blocks), dtype=np.int32)
        pos = 0
        for s, n in enumerate(nblk):
            self.tables[s, :n] = perm[pos:pos + n]
            pos += n
        self.k_f32 = [synth.normal_f32(seed, (200 << 32) | s, int(c) * hkv * d).reshape(-1, hkv, d)
                      for s, c in enumerate(self.ctx)]
        self.v_f32 = [synth.normal_f32(seed, (300 << 32) | s, int(c) * hkv * d).reshape(-1, hkv, d)
                      for s, c in enumerate(self.ctx)]
        self.q_store = workloads.cast(synth.normal_f32(seed, 400, batch * hq * d).reshape(batch, hq, d), q_dtype)
        self.k_src = [workloads.cast(x, self.src_dtype) for x in self.k_f32]
        self.v_src = [workloads.cast(x, self.src_dtype) for x in self.v_f32]
        if kv_dtype == "fp8_e4m3":
            allk = np.concatenate([numerics.source_to_f32(x, self.src_dtype).ravel() for x in self.k_src] + [np.zeros(1, np.float32)])
            allv = np.concatenate([numerics.source_to_f32(x, self.src_dtype).ravel() for x in self.v_src] + [np.zeros(1, np.float32)])
            self.k_scale = float(max(workloads.fp8_scale_of(allk), np.float32(1e-3)))
            self.v_scale = float(max(workloads.fp8_scale_of(allv), np.float32(1e-3)))
        else:
            self.k_scale = self.v_scale = 1.0
        self.scale = 1.0 / math.sqrt(d)

    def desc(self, pa):
        return pa.CacheDesc(self.num_blocks, self.bs, self.hkv, self.d, self.kv_dtype, self.k_scale, self.v_scale)

    def seq_pos(self):
        seq = np.concatenate([np.full(int(c), s, dtype=np.int32) for s, c in enumerate(self.ctx)] + [np.zeros(0, np.int32)])
        pos = np.concatenate([np.arange(int(c), dtype=np.int32) for c in self.ctx] + [np.zeros(0, np.int32)])
        return seq, pos

    # ---- library side
    def gpu_pools(self, pa, device, status=None):
        desc = self.desc(pa)
        kc, vc = desc.new_pools(device, fill=POISON)
        seq, pos = self.seq_pos()
        if len(seq):
            slots = pa.compute_slot_mapping(self.tables, seq, pos, self.bs)
            k = to_torch(np.concatenate(self.k_src), self.src_dtype, device)
            v = to_torch(np.concatenate(self.v_src), self.src_dtype, device)
            pa.kv_append(desc, k, v, torch.from_numpy(slots).to(device), kc, vc, status=status)
        return kc, vc

    def gpu_decode(self, pa, device, kc, vc, out_dtype="f32", partition=None, status=None):
        q = to_torch(self.q_store, self.q_dtype, device)
        bt = torch.from_numpy(self.tables).to(device)
        cl = torch.from_numpy(self.ctx).to(device)
        part = self.partition if partition is None else partition
        return pa.decode_attention(self.desc(pa), q, kc, vc, bt, cl, self.scale, partition=part,
                                   out_dtype=out_dtype, status=status)

    # ---- oracle side
    def oracle_pools(self):
        kp = ocache.new_pool(self.num_blocks, self.hkv, self.bs, self.d, self.kv_dtype, fill=0)
        vp = ocache.new_pool(self.num_blocks, self.hkv, self.bs, self.d, self.kv_dtype, fill=0)
        kp.view(np.uint8)[...] = POISON
        vp.view(np.uint8)[...] = POISON
        seq, pos = self.seq_pos()
        if len(seq):
            slots = ocache.slot_mapping(self.tables, seq, pos, self.bs)
            ocache.kv_append(kp, vp, np.concatenate(self.k_src), np.concatenate(self.v_src), slots,
                             self.src_dtype, self.kv_dtype, self.k_scale, self.v_scale)
        return kp, vp

    def oracle_out(self, kp, vp):
        return oatt.decode_attention_paged(self.q_store, kp, vp, self.tables, self.ctx, self.scale, self.kv_dtype,
                                           self.k_scale, self.v_scale, q_dtype=self.q_dtype)


def assert_close(got, expect, tol, what=""):
    got = np.asarray(got, dtype=np.float64)
    err = np.abs(got - expect)
    worst = float(np.max(err)) if err.size else 0.0
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert worst <= tol, f"{what}: max abs error {worst:.3e} > {tol:.1e}"
    return worst

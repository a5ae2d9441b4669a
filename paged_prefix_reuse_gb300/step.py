"""One step of the hot path on the GPU: copy-on-write forks, slot indexing,
append of the new tokens' K/V, prefix attention for the prefill chunks and
decode attention for the decode batch -- all through libkvp's C ABI.

``DeviceStep`` takes any object with the attributes of a workload (numpy
arrays of bit patterns and int32 tables; see ``workloads.Workload``), moves
them to the device once, and ``run()`` enqueues the whole step on a stream.
The sequences are ordered prefill chunks first, then ``num_decode`` decode
sequences with one new token each.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (
    PagedKVPool,
    kvp_block_copy,
    kvp_cache_append,
    kvp_decode_attn,
    kvp_decode_num_splits,
    kvp_prefix_attn,
    kvp_prefix_num_splits,
    kvp_slot_mapping,
    kvp_workspace_size,
)

_TORCH_DT = {"f16": torch.float16, "bf16": torch.bfloat16}


def bits_to_device(bits: np.ndarray, dtype: str, device) -> torch.Tensor:
    """uint16 bit patterns -> a device tensor of the storage dtype (same bytes)."""
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.to(device).view(_TORCH_DT[dtype])


class DeviceStep:
    def __init__(self, w, device="cuda", prefix_splits: int = 0, decode_splits: int = 0):
        self.w = w
        self.device = torch.device(device)
        dev = self.device
        self.pool = PagedKVPool(bits_to_device(w.k_pool, w.dtype, dev), bits_to_device(w.v_pool, w.dtype, dev))
        self.q = bits_to_device(w.q, w.dtype, dev)
        self.k_new = bits_to_device(w.k_new, w.dtype, dev)
        self.v_new = bits_to_device(w.v_new, w.dtype, dev)
        cu = np.asarray(w.cu_seqlens_q, dtype=np.int32)
        ctx = np.asarray(w.context_lens, dtype=np.int32)
        bt = np.ascontiguousarray(w.block_tables, dtype=np.int32)
        self.cu = torch.from_numpy(cu).to(dev)
        self.ctx = torch.from_numpy(ctx).to(dev)
        self.bt = torch.from_numpy(bt).to(dev)
        self.pairs = torch.from_numpy(np.ascontiguousarray(w.cow_pairs, dtype=np.int32).reshape(-1, 2)).to(dev)
        self.T = int(cu[-1])
        self.slots = torch.empty(max(self.T, 1), dtype=torch.int64, device=dev)
        B = int(ctx.shape[0])
        self.npf = B - int(w.num_decode)
        self.ndec = int(w.num_decode)
        Hq, Hkv, d = w.num_q_heads, w.num_kv_heads, w.head_dim
        self.scale = float(w.softmax_scale)
        new_lens = np.diff(cu)
        # prefill sub-batch: sequences [0, npf)
        self.tq = int(cu[self.npf])
        if self.npf > 0:
            self.max_q_pf = int(new_lens[: self.npf].max()) if self.npf else 0
            self.max_ctx_pf = int(ctx[: self.npf].max())
            self.prefix_splits = prefix_splits or kvp_prefix_num_splits(
                self.npf, Hq, Hkv, d, max(self.max_q_pf, 1), max(self.max_ctx_pf, 1))
            self.out_pf = torch.empty((self.tq, Hq, d), dtype=self.q.dtype, device=dev)
            self.lse_pf = torch.empty((Hq, self.tq), dtype=torch.float32, device=dev)
            need = kvp_workspace_size(0, self.tq, Hq, d, self.prefix_splits)
            self.ws_pf = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        if self.ndec > 0:
            self.max_ctx_dec = int(ctx[self.npf :].max())
            self.decode_splits = decode_splits or kvp_decode_num_splits(
                self.ndec, Hkv, w.block_size, self.max_ctx_dec)
            self.out_dec = torch.empty((self.ndec, Hq, d), dtype=self.q.dtype, device=dev)
            self.lse_dec = torch.empty((Hq, self.ndec), dtype=torch.float32, device=dev)
            need = kvp_workspace_size(1, self.ndec, Hq, d, self.decode_splits)
            self.ws_dec = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)

    # ---- the individual calls (used for per-kernel timing) ----
    def run_copy(self, stream=None):
        if self.pairs.shape[0]:
            kvp_block_copy(self.pool, self.pairs, stream=stream)

    def run_slots(self, stream=None):
        if self.T:
            kvp_slot_mapping(self.pool, self.cu, self.ctx, self.bt, self.T, out=self.slots, stream=stream)

    def run_append(self, stream=None):
        if self.T:
            kvp_cache_append(self.pool, self.k_new, self.v_new, self.slots[: self.T], stream=stream)

    def run_prefill(self, stream=None):
        if self.npf > 0 and self.tq > 0:
            kvp_prefix_attn(self.pool, self.q[: self.tq], self.cu[: self.npf + 1], self.ctx[: self.npf],
                            self.bt[: self.npf], self.max_q_pf, self.max_ctx_pf, self.scale,
                            num_splits=self.prefix_splits, out=self.out_pf, lse=self.lse_pf,
                            workspace=self.ws_pf, stream=stream)

    def run_decode(self, stream=None):
        if self.ndec > 0:
            kvp_decode_attn(self.pool, self.q[self.tq :], self.ctx[self.npf :], self.bt[self.npf :],
                            self.max_ctx_dec, self.scale, num_splits=self.decode_splits, out=self.out_dec,
                            lse=self.lse_dec, workspace=self.ws_dec, stream=stream)

    def run(self, stream=None):
        """Enqueue the whole step on ``stream`` (default: current stream)."""
        self.run_copy(stream)
        self.run_slots(stream)
        self.run_append(stream)
        self.run_prefill(stream)
        self.run_decode(stream)

    def reset_pool(self):
        """Restore the pool contents the workload started with."""
        self.pool.k.copy_(bits_to_device(self.w.k_pool, self.w.dtype, self.device))
        self.pool.v.copy_(bits_to_device(self.w.v_pool, self.w.dtype, self.device))

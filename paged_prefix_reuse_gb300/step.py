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


class HostStep:
    """The step from pinned host buffers, with its transfers overlapped.

    The inputs (q, the new K/V, the tables and the copy-on-write pairs) sit in
    pinned host memory and the outputs (O and LSE) go back to pinned host
    memory.  The prefill sequences are split into ``groups`` contiguous
    ranges of about equal token counts (0: one group per GPU's worth of
    prefix-attention CTAs, see ``auto_groups``) and the decode batch forms one more
    group; each group runs on its own stream as host->device copy of its
    tokens, slot mapping, append, attention and device->host copy of its
    outputs, so one group's copies overlap another group's kernels and the
    two copy directions overlap each other.  The tables of all groups travel
    in one copy on ``stream``, followed by the copy-on-write block copies;
    every group's kernels wait for both.  Groups share no pool block they write (a write
    goes only into a block its sequence owns alone), so their order does not
    matter.

    The groups' calls are the library calls the one-stream step makes, on
    slices of the same device buffers; with the same split counts the
    outputs are bit-identical to ``DeviceStep.run``.  LSE comes back per
    group (``lse_host[i]`` is [Hq, tokens of group i]).
    """

    def __init__(self, st: DeviceStep, groups: int = 0, prefix_splits: int = 0, decode_splits: int = 0):
        self.st = st
        w = st.w
        dev = st.device
        cu = np.asarray(w.cu_seqlens_q, dtype=np.int64)
        ctx = np.asarray(w.context_lens, dtype=np.int32)
        bt = np.ascontiguousarray(w.block_tables, dtype=np.int32)
        mb = int(bt.shape[1])
        Hq, d = w.num_q_heads, w.head_dim
        if groups <= 0:
            groups = self.auto_groups(w, st.npf)
        plan = self.plan(cu, st.npf, st.ndec, groups)

        parts, off = [], 0

        def put(a):
            nonlocal off
            a = np.ascontiguousarray(a, dtype=np.int32).ravel()
            start = off
            pad = (-a.size) % 4  # 16-byte aligned starts
            parts.append(np.concatenate([a, np.zeros(pad, dtype=np.int32)]))
            off += a.size + pad
            return start, a.size

        self.groups = []
        for kind, a, b, c0, c1 in plan:
            if c0 is None:  # whole sequences [a, b)
                g = {"kind": kind, "n": b - a, "t0": int(cu[a]), "t1": int(cu[b]), "chunk": False,
                     "cu": put(cu[a : b + 1] - cu[a]), "ctx": put(ctx[a:b]), "bt": put(bt[a:b]),
                     "max_q": int(np.diff(cu[a : b + 1]).max()), "max_ctx": int(ctx[a:b].max())}
            else:  # new tokens [c0, c1) of sequence a: its keys end at P + c1
                n_new = int(cu[a + 1] - cu[a])
                cend = int(ctx[a]) - (n_new - c1)
                g = {"kind": kind, "n": 1, "t0": int(cu[a]) + c0, "t1": int(cu[a]) + c1, "chunk": c0 > 0,
                     "cu": put([0, c1 - c0]), "ctx": put([cend]), "bt": put(bt[a : a + 1]),
                     "max_q": c1 - c0, "max_ctx": cend}
            self.groups.append(g)
        meta = np.concatenate(parts) if parts else np.zeros(4, dtype=np.int32)
        self.h_meta = torch.from_numpy(meta).pin_memory()
        self.d_meta = torch.empty(meta.shape, dtype=torch.int32, device=dev)
        for g in self.groups:
            n, T = g["n"], g["t1"] - g["t0"]
            g["d_cu"] = self.d_meta[g["cu"][0] : g["cu"][0] + n + 1]
            g["d_ctx"] = self.d_meta[g["ctx"][0] : g["ctx"][0] + n]
            g["d_bt"] = self.d_meta[g["bt"][0] : g["bt"][0] + n * mb].view(n, mb)
            g["lse"] = torch.empty((Hq, T), dtype=torch.float32, device=dev)
            g["lse_host"] = torch.empty((Hq, T), dtype=torch.float32).pin_memory()
            if g["kind"] == "prefill":
                g["splits"] = prefix_splits or st.prefix_splits
                need = kvp_workspace_size(0, T, Hq, d, g["splits"])
            else:
                g["splits"] = decode_splits or st.decode_splits
                need = kvp_workspace_size(1, T, Hq, d, g["splits"])
            g["ws"] = torch.empty(max(need, 1), dtype=torch.uint8, device=dev)
        self.lse_host = [g["lse_host"] for g in self.groups]
        self.h_q = st.q.cpu().pin_memory()
        self.h_k = st.k_new.cpu().pin_memory()
        self.h_v = st.v_new.cpu().pin_memory()
        self.h_pairs = st.pairs.cpu().pin_memory()
        self.out_host = torch.empty(st.q.shape, dtype=st.q.dtype).pin_memory()  # O of every token
        self.streams = [torch.cuda.Stream(device=dev) for _ in self.groups]
        self.h2d_bytes = sum(t.numel() * t.element_size() for t in (self.h_meta, self.h_q, self.h_k, self.h_v,
                                                                     self.h_pairs))
        self.d2h_bytes = self.out_host.numel() * self.out_host.element_size() + sum(
            g["lse_host"].numel() * 4 for g in self.groups)

    @staticmethod
    def plan(cu_seqlens_q, npf: int, ndec: int, groups: int, align: int = 256):
        """[(kind, a, b, c0, c1)]: with no more groups than prefill sequences
        that have new tokens, ``partition``'s ranges of whole sequences [a, b)
        (c0 = c1 = None); with more, each such sequence a's new tokens cut into
        ceil(groups / sequences) chunks [c0, c1) of about equal length, in
        multiples of ``align`` tokens (one group each), then the decode batch.
        A chunk's queries see the keys up to its own end, so its call needs
        the earlier chunks' K/V appended first."""
        cu = np.asarray(cu_seqlens_q, dtype=np.int64)
        live = [s for s in range(npf) if cu[s + 1] > cu[s]]
        if groups <= len(live):
            return [(k, a, b, None, None) for k, a, b in HostStep.partition(cu, npf, ndec, groups)]
        per = -(-groups // len(live))
        out = []
        for s in live:
            n = int(cu[s + 1] - cu[s])
            chunk = -(-n // per)  # ceil(n / per)
            step = max(align, -(-chunk // align) * align)  # rounded up to whole multiples of align
            c0 = 0
            while c0 < n:
                c1 = min(n, c0 + step)
                out.append(("prefill", s, s + 1, c0, c1))
                c0 = c1
        if ndec:
            out.append(("decode", npf, npf + ndec, None, None))
        return out

    @staticmethod
    def partition(cu_seqlens_q, npf: int, ndec: int, groups: int):
        """[(kind, first sequence, end sequence)]: the prefill sequences [0, npf)
        cut into at most ``groups`` contiguous ranges of about equal token
        counts (ranges without tokens dropped), then the decode batch."""
        cu = np.asarray(cu_seqlens_q, dtype=np.int64)
        ranges = []
        if npf and cu[npf] > 0:
            tq = int(cu[npf])
            bounds = [0]
            for k in range(1, max(1, groups)):
                s = int(np.searchsorted(cu[1 : npf + 1], tq * k / groups)) + 1
                bounds.append(min(max(s, bounds[-1]), npf))
            bounds.append(npf)
            ranges = [("prefill", a, b) for a, b in zip(bounds[:-1], bounds[1:]) if cu[b] > cu[a]]
        if ndec:
            ranges.append(("decode", npf, npf + ndec))
        return ranges

    @staticmethod
    def auto_groups(w, npf: int, sms: int = 152, rows_per_cta: int = 256, most: int = 16) -> int:
        """One group per GPU's worth of prefix-attention CTAs, or one per
        prefill sequence that fills at least half the GPU alone, whichever is
        more (at most ``most``).  A group that leaves most SMs idle gains
        little from starting early, and each group adds its own launches and
        copies.  Measured (e2e TFLOP/s by prefill groups): the mixed batch
        (four sequences of 80 CTAs) 308 at 2, 357 at 4, 300 at 8; the RAG
        batch (sixteen of 42) 162 at 2, 207 at 4, 189 at 8."""
        if npf <= 0:
            return 1
        g = w.num_q_heads // w.num_kv_heads
        n = np.diff(np.asarray(w.cu_seqlens_q, dtype=np.int64))[:npf]
        per_seq = ((n * g + rows_per_cta - 1) // rows_per_cta) * w.num_kv_heads
        big = int(np.sum(2 * per_seq >= sms))
        return max(1, min(most, max(int(per_seq.sum()) // sms, big)))

    def run(self, stream=None):
        """Enqueue the step; everything is ordered before work later queued on
        ``stream`` (default: current stream).  The host outputs are complete
        once that stream has passed this point."""
        st = self.st
        s0 = stream if stream is not None else torch.cuda.current_stream()
        # Every group stream first follows ``stream`` (in a graph capture, this
        # is how a side stream joins the capture).
        fork = torch.cuda.Event()
        fork.record(s0)
        with torch.cuda.stream(s0):
            self.d_meta.copy_(self.h_meta, non_blocking=True)
            if st.pairs.shape[0]:
                st.pairs.copy_(self.h_pairs, non_blocking=True)
                kvp_block_copy(st.pool, st.pairs, stream=s0)
        ready = torch.cuda.Event()
        ready.record(s0)
        done = []
        landed = None  # the previous group's host-to-device copies
        appended = []  # each earlier group's appends
        for g, s in zip(self.groups, self.streams):
            t0, t1 = g["t0"], g["t1"]
            s.wait_event(fork)
            with torch.cuda.stream(s):
                # The group's tokens need no table, so their copies start at
                # once -- but after the previous group's: the copies share one
                # host link, and in group order the first group's kernels start
                # after its own share of the bytes instead of after all of them.
                if landed is not None:
                    s.wait_event(landed)
                st.q[t0:t1].copy_(self.h_q[t0:t1], non_blocking=True)
                st.k_new[t0:t1].copy_(self.h_k[t0:t1], non_blocking=True)
                st.v_new[t0:t1].copy_(self.h_v[t0:t1], non_blocking=True)
                landed = torch.cuda.Event()
                landed.record(s)
                s.wait_event(ready)
                kvp_slot_mapping(st.pool, g["d_cu"], g["d_ctx"], g["d_bt"], t1 - t0, out=st.slots[t0:t1], stream=s)
                kvp_cache_append(st.pool, st.k_new[t0:t1], st.v_new[t0:t1], st.slots[t0:t1], stream=s)
                if g["chunk"]:
                    # A later chunk of a sequence attends to the K/V the
                    # earlier chunks' groups append.
                    for e in appended:
                        s.wait_event(e)
                ea = torch.cuda.Event()
                ea.record(s)
                appended.append(ea)
                if g["kind"] == "prefill":
                    out = st.out_pf[t0:t1]
                    kvp_prefix_attn(st.pool, st.q[t0:t1], g["d_cu"], g["d_ctx"], g["d_bt"], g["max_q"], g["max_ctx"],
                                    st.scale, num_splits=g["splits"], out=out, lse=g["lse"], workspace=g["ws"],
                                    stream=s)
                else:
                    out = st.out_dec
                    kvp_decode_attn(st.pool, st.q[t0:t1], g["d_ctx"], g["d_bt"], g["max_ctx"], st.scale,
                                    num_splits=g["splits"], out=out, lse=g["lse"], workspace=g["ws"], stream=s)
                self.out_host[t0:t1].copy_(out, non_blocking=True)
                g["lse_host"].copy_(g["lse"], non_blocking=True)
            e = torch.cuda.Event()
            e.record(s)
            done.append(e)
        for e in done:
            s0.wait_event(e)

    def capture(self, stream) -> torch.cuda.CUDAGraph:
        """The step as one CUDA graph, copies included: each replay moves the
        current contents of the pinned inputs in, runs every group and moves
        the outputs out, with no host work per step.  ``stream`` is the
        capture (and replay-ordering) stream."""
        self.run(stream)  # once outside capture: the library's one-time setup
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            self.run(stream)
        return graph

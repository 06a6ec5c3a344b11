"""Drive the C ABI from a synthetic workload: build the cache, batch and plan.

Everything here is argument marshalling around ``binding``: the workload's
op list is replayed through ``kv_branch_create`` / ``kv_append`` /
``kv_fork_branches`` / ``kv_evict``, the decode batch comes from
``kv_build_batch`` and the work split from ``paged_decode_plan``; torch only
allocates device memory and uploads host arrays.  With ``with_data=False``
the pool is metadata-only (no device memory, no kernels): that is how the
allocator is exercised on a machine without a GPU.
"""

from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import binding as B


def _to_device_bf16(a: np.ndarray, device):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16))
    return t.to(device).view(torch.bfloat16)


class Cache:
    """A pool holding one workload's tree, built through the C ABI."""

    def __init__(self, w, with_data: bool = True, device: str = "cuda",
                 evict: bool = True, kv_dtype: str = "bf16",
                 poison: bool = False, replay: bool = True):
        """kv_dtype: "bf16" or "e4m3" (codes [L][blocks][Hkv][16 * d] uint8
        plus scale records [L][blocks][Hkv][4] float32).  poison: fill the
        pools with NaN (bf16 NaN, e4m3 NaN codes and NaN scales) before any
        write.  replay=False: create the pool only (no ops, no eviction)."""
        self.w = w
        self.with_data = with_data
        self.device = device
        self.kv_dtype = kv_dtype
        self.e4m3 = kv_dtype == "e4m3"
        if kv_dtype not in ("bf16", "e4m3"):
            raise ValueError(kv_dtype)
        self.k = self.v = self.scales = None
        if with_data:
            import torch
            if self.e4m3:
                shape = (w.num_layers, w.num_blocks, w.Hkv, w.block_size * w.d)
                self.k = torch.empty(shape, dtype=torch.uint8, device=device)
                self.v = torch.empty(shape, dtype=torch.uint8, device=device)
                self.scales = torch.zeros(
                    (w.num_layers, w.num_blocks, w.Hkv, 4),
                    dtype=torch.float32, device=device)
                if poison:
                    self.k.fill_(0x7F)
                    self.v.fill_(0x7F)
                    self.scales.fill_(float("nan"))
            else:
                shape = (w.num_layers, w.num_blocks, w.Hkv, w.block_size, w.d)
                self.k = torch.empty(shape, dtype=torch.bfloat16, device=device)
                self.v = torch.empty(shape, dtype=torch.bfloat16, device=device)
                if poison:
                    self.k.fill_(float("nan"))
                    self.v.fill_(float("nan"))
        self.h = B.kv_pool_create(
            w.num_blocks, w.num_layers, w.Hkv, w.d, self.k, self.v,
            w.initial_free_order(), w.block_size,
            B.KV_DTYPE_E4M3 if self.e4m3 else B.KV_DTYPE_BF16, self.scales)
        self.evicted: list = []
        self.decode_ids: list = []
        if not replay:
            return
        self._replay()
        if evict and w.evict_target_leaves() > 0:
            cand = w.evict_candidates()
            self.evicted = B.kv_evict(self.h, cand,
                                      [w.evict_scores[i] for i in cand],
                                      B.KV_STOP_EVICTED_LEAVES,
                                      w.evict_target_leaves())
        self.decode_ids = [i for i in w.leaves()
                           if B.kv_branch_info(self.h, i)["live"]]

    def _replay(self):
        w = self.w
        for op in w.ops:
            if op[0] == "create":
                nid = B.kv_branch_create(self.h)
                if nid >= len(w.nodes) or w.nodes[nid].parent != -1:
                    raise RuntimeError("handle order differs from the workload")
            elif op[0] == "append":
                nid = op[1]
                n = w.nodes[nid].n_tokens
                if self.with_data:
                    k, v = w.node_kv(nid)
                    kd = _to_device_bf16(k, self.device)
                    vd = _to_device_bf16(v, self.device)
                    B.kv_append(self.h, nid, n, kd, vd)
                else:
                    B.kv_append(self.h, nid, n)
            elif op[0] == "fork":
                kids = B.kv_fork_branches(self.h, op[1], op[2])
                for c in kids:
                    if w.nodes[c].parent != op[1]:
                        raise RuntimeError("fork order differs from the workload")
            else:
                raise ValueError(op)

    def close(self):
        if self.h is not None:
            B.kv_pool_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- state for bit-exact comparison --------------------------------------
    def tables(self) -> dict:
        out = {}
        for i in range(B.kv_num_branches(self.h)):
            info = B.kv_branch_info(self.h, i)
            if info["live"]:
                t, L = B.kv_get_block_table(self.h, i)
                out[i] = (t.tolist(), L)
        return out

    def refcounts(self) -> list:
        return B.kv_get_refcounts(self.h, self.w.num_blocks).tolist()

    def free_stack(self) -> list:
        return B.kv_get_free_stack(self.h).tolist()

    # -- decode ----------------------------------------------------------------
    def batch(self, ids=None, flags: int = 0, num_sms: int = 0) -> "Batch":
        ids = self.decode_ids if ids is None else list(ids)
        tables, lens, groups = B.kv_build_batch(self.h, ids)
        nb, max_blocks = tables.shape
        if num_sms == 0 and self.with_data:
            import torch
            num_sms = torch.cuda.get_device_properties(
                self.device).multi_processor_count
        if self.e4m3:
            flags |= B.KV_PLAN_KV_E4M3
        plan, info = B.paged_decode_plan(nb, self.w.Hq, self.w.Hkv, self.w.d,
                                         max_blocks, lens, groups, num_sms,
                                         flags, self.w.block_size)
        return Batch(self, ids, tables, lens, groups, plan, info)


@dataclass
class Batch:
    cache: Cache
    ids: list
    tables: np.ndarray
    seq_lens: np.ndarray
    groups: np.ndarray
    plan: np.ndarray
    info: object
    dev: dict = None

    def upload(self):
        import torch
        dev = self.cache.device
        self.dev = {
            "tables": torch.from_numpy(self.tables).to(dev),
            "seq_lens": torch.from_numpy(self.seq_lens).to(dev),
            "groups": torch.from_numpy(np.ascontiguousarray(
                self.groups.reshape(-1)) if len(self.groups)
                else np.zeros(4, np.int32)).to(dev),
            "plan": torch.from_numpy(self.plan).to(dev),
            "workspace": torch.empty(max(self.info.workspace_bytes, 256),
                                     dtype=torch.uint8, device=dev),
        }
        return self

    @property
    def nb(self) -> int:
        return len(self.ids)

    def decode(self, q, out, layer: int = 0, stream=None):
        """q, out: device bf16 [nb][Hq][d]."""
        c = self.cache
        w = c.w
        if self.dev is None:
            self.upload()
        d = self.dev
        if c.e4m3:
            B.paged_decode_attn_e4m3(
                q, c.k[layer], c.v[layer], c.scales[layer], w.num_blocks,
                d["tables"], d["seq_lens"], d["groups"], len(self.groups),
                self.nb, self.tables.shape[1], w.Hq, w.Hkv, w.d, w.scale, out,
                d["plan"], self.info, d["workspace"], d["workspace"].numel(),
                stream, w.block_size)
            return
        B.paged_decode_attn(q, c.k[layer], c.v[layer], w.num_blocks,
                            d["tables"], d["seq_lens"], d["groups"],
                            len(self.groups), self.nb, self.tables.shape[1],
                            w.Hq, w.Hkv, w.d, w.scale, out, d["plan"],
                            self.info, d["workspace"], d["workspace"].numel(),
                            stream, w.block_size)

    def decode_append(self, q, k_step, v_step, out, layer: int = 0,
                      stream=None):
        """Decode step that also writes each branch's newest token (reserved
        beforehand with kv_reserve): k_step, v_step device bf16 [nb][Hkv][d]."""
        c = self.cache
        w = c.w
        if self.dev is None:
            self.upload()
        d = self.dev
        if c.e4m3:
            B.paged_decode_append_attn_e4m3(
                q, k_step, v_step, c.k[layer], c.v[layer], c.scales[layer],
                w.num_blocks, d["tables"], d["seq_lens"], d["groups"],
                len(self.groups), self.nb, self.tables.shape[1], w.Hq, w.Hkv,
                w.d, w.scale, out, d["plan"], self.info, d["workspace"],
                d["workspace"].numel(), stream, w.block_size)
            return
        B.paged_decode_append_attn(q, k_step, v_step, c.k[layer], c.v[layer],
                                   w.num_blocks, d["tables"], d["seq_lens"],
                                   d["groups"], len(self.groups), self.nb,
                                   self.tables.shape[1], w.Hq, w.Hkv, w.d,
                                   w.scale, out, d["plan"], self.info,
                                   d["workspace"], d["workspace"].numel(),
                                   stream, w.block_size)

    def device_status(self, stream=None):
        return B.kv_check_device_status(self.dev["workspace"], stream)

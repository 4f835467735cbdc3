"""Puts a seeded workload on the GPU and runs it through the C ABI.

Shared by the GPU tests, bench.py and __graft_entry__.smoke().  It allocates
device memory with torch (inputs, sentinel-filled destination pools, block
tables, the batch workspace) and calls the library entry point that fits the
workload: kv_relocate_patch (or _mrope) for one GQA/MHA chunk,
kv_relocate_patch_mla for one MLA chunk, and for several chunks
kv_relocate_batch, kv_relocate_batch_mrope or kv_relocate_batch_mla.  No
arithmetic of the operator happens here.
"""
from __future__ import annotations

import numpy as np
import torch

import position_invariant_kv_gb300 as kvrp
import workloads as W

SENTINEL = -1  # int16 view of 0xFFFF, a bf16 NaN pattern no result can take


def _bf16(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(device).view(torch.bfloat16)


class DeviceWorkload:
    """Inputs, pools and launch arguments of one workload on one device."""

    def __init__(self, wl: W.Workload, device="cuda", host=None):
        self.wl = wl
        self.device = torch.device(device)
        if wl.backend == "numpy" or host is not None:
            host = host if host is not None else W.host_inputs(wl)
            self.host = host
            self.rows = {n: _bf16(host["rows"][n], self.device) for n in wl.tensors}
            self.u = {n: [None if a is None else _bf16(a, self.device) for a in host["u"][n]] for n in wl.tensors}
            self.w = {n: [None if a is None else _bf16(a, self.device) for a in host["w"][n]] for n in wl.tensors}
        else:
            self.host = None
            d = W.torch_inputs(wl, str(self.device))
            self.rows, self.u, self.w = d["rows"], d["u"], d["w"]
        self.block_tables = None
        if wl.paged:
            self.block_tables = torch.from_numpy(np.ascontiguousarray(wl.block_tables, np.int32)).to(self.device)
        D = wl.row_width
        self.pools = {n: torch.empty((wl.n_layers, wl.num_pages, W.PAGE, D), dtype=torch.bfloat16,
                                     device=self.device) for n in wl.tensors}
        self.reset_pools()
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)
        self.workspace = None
        if len(wl.chunks) > 1:
            nbytes = kvrp.kv_relocate_batch_workspace_size(len(wl.chunks))
            self.workspace = torch.empty(nbytes, dtype=torch.uint8, device=self.device)
        self._chunks = self._chunk_args()
        self._batch_array = None

    def replica(self) -> "DeviceWorkload":
        """A second device copy of this workload (inputs, pools, status,
        workspace), with launch arguments pointing at the copy."""
        r = object.__new__(DeviceWorkload)
        r.wl, r.device, r.host = self.wl, self.device, self.host
        r.rows = {n: t.clone() for n, t in self.rows.items()}
        r.u = {n: [None if t is None else t.clone() for t in ts] for n, ts in self.u.items()}
        r.w = {n: [None if t is None else t.clone() for t in ts] for n, ts in self.w.items()}
        r.block_tables = None if self.block_tables is None else self.block_tables.clone()
        r.pools = {n: p.clone() for n, p in self.pools.items()}
        r.status = torch.zeros_like(self.status)
        r.workspace = None if self.workspace is None else torch.empty_like(self.workspace)
        r._chunks = r._chunk_args()
        r._batch_array = None
        return r

    def reset_pools(self):
        for p in self.pools.values():
            p.view(torch.int16).fill_(SENTINEL)

    def _dst(self, name, c: W.Chunk) -> kvrp.Dst:
        wl = self.wl
        pool = self.pools[name]
        bt = None
        if wl.paged:
            bt = self.block_tables[c.seq]
        return kvrp.Dst(base=pool, num_pages=wl.num_pages, layer_stride=pool.stride(0),
                        block_table=bt, dst_start=c.dst_start)

    def _src(self, name, c: W.Chunk) -> int:
        t = self.rows[name]
        return t.data_ptr() + c.src_row0 * t.stride(1) * t.element_size()

    def _chunk_args(self):
        wl = self.wl
        out = []
        for ci, c in enumerate(wl.chunks):
            a = {"n_tokens": c.n_tokens, "delta": c.delta, "rank": c.rank}
            names = wl.tensors
            a["srcs"] = [self._src(n, c) for n in names]
            a["src_layer_stride"] = self.rows[names[0]].stride(0)
            a["u"] = [self.u[n][ci] for n in names]
            a["w"] = [self.w[n][ci] for n in names]
            a["u_layer_stride"] = c.n_tokens * c.rank
            a["w_layer_stride"] = wl.row_width * c.rank
            a["dst"] = [self._dst(n, c) for n in names]
            out.append(a)
        return out

    def launch_count(self) -> int:
        return 1

    def run(self, stream=None):
        """One pass of the whole operator over the workload (one kernel launch)."""
        wl = self.wl
        if wl.family == "mla" and len(wl.chunks) > 1:
            if self._batch_array is None:
                self._batch_array = kvrp.mla_chunk_array(self.mla_batch_chunks())
            kvrp.kv_relocate_batch_mla(self._batch_array, n_layers=wl.n_layers, kv_lora_dim=wl.kv_lora_dim,
                                       rope_dim=wl.rope_dim, rope_theta=wl.theta, workspace=self.workspace,
                                       d_status=self.status, stream=stream)
        elif wl.family == "mla":
            a = self._chunks[0]
            kvrp.kv_relocate_patch_mla(
                a["srcs"][0], n_layers=wl.n_layers, n_tokens=a["n_tokens"], kv_lora_dim=wl.kv_lora_dim,
                rope_dim=wl.rope_dim, delta=a["delta"], rope_theta=wl.theta, dst=a["dst"][0],
                rank=a["rank"], u=a["u"][0], v=a["w"][0], src_layer_stride=a["src_layer_stride"],
                u_layer_stride=a["u_layer_stride"], v_layer_stride=a["w_layer_stride"],
                d_status=self.status, stream=stream)
        elif len(wl.chunks) == 1 and wl.mrope_sections is not None:
            a = self._chunks[0]
            kvrp.kv_relocate_patch_mrope(
                a["srcs"][0], a["srcs"][1], n_layers=wl.n_layers, n_tokens=a["n_tokens"],
                n_kv_heads=wl.n_heads, head_dim=wl.head_dim, delta_thw=a["delta"],
                mrope_section=wl.mrope_sections, rope_theta=wl.theta,
                k_dst=a["dst"][0], v_dst=a["dst"][1], rank=a["rank"], uk=a["u"][0], vk=a["w"][0],
                uv=a["u"][1], vv=a["w"][1], src_layer_stride=a["src_layer_stride"],
                u_layer_stride=a["u_layer_stride"], v_layer_stride=a["w_layer_stride"],
                d_status=self.status, stream=stream)
        elif len(wl.chunks) == 1:
            a = self._chunks[0]
            kvrp.kv_relocate_patch(
                a["srcs"][0], a["srcs"][1], n_layers=wl.n_layers, n_tokens=a["n_tokens"],
                n_kv_heads=wl.n_heads, head_dim=wl.head_dim, delta=a["delta"], rope_theta=wl.theta,
                k_dst=a["dst"][0], v_dst=a["dst"][1], rank=a["rank"], uk=a["u"][0], vk=a["w"][0],
                uv=a["u"][1], vv=a["w"][1], src_layer_stride=a["src_layer_stride"],
                u_layer_stride=a["u_layer_stride"], v_layer_stride=a["w_layer_stride"],
                d_status=self.status, stream=stream)
        elif wl.mrope_sections is not None:
            if self._batch_array is None:
                self._batch_array = kvrp.chunk_array(self.batch_chunks())
            kvrp.kv_relocate_batch_mrope(self._batch_array, [a["delta"] for a in self._chunks], n_layers=wl.n_layers,
                                         n_kv_heads=wl.n_heads, head_dim=wl.head_dim,
                                         mrope_section=wl.mrope_sections, rope_theta=wl.theta,
                                         workspace=self.workspace, d_status=self.status, stream=stream)
        else:
            if self._batch_array is None:            # the chunks do not change: marshal them once
                self._batch_array = kvrp.chunk_array(self.batch_chunks())
            kvrp.kv_relocate_batch(self._batch_array, n_layers=wl.n_layers, n_kv_heads=wl.n_heads,
                                   head_dim=wl.head_dim, rope_theta=wl.theta, workspace=self.workspace,
                                   d_status=self.status, stream=stream)

    def mla_batch_chunks(self) -> list:
        """The workload's chunks as kv_relocate_batch_mla descriptors."""
        return [kvrp.MlaChunk(src=a["srcs"][0], n_tokens=a["n_tokens"], delta=a["delta"], dst=a["dst"][0],
                              rank=a["rank"], u=a["u"][0], v=a["w"][0], src_layer_stride=a["src_layer_stride"],
                              u_layer_stride=a["u_layer_stride"], v_layer_stride=a["w_layer_stride"])
                for a in self._chunks]

    def batch_chunks(self) -> list:
        """The workload's chunks as kv_relocate_batch descriptors (under M-RoPE
        the .delta field is unused: the (t, h, w) shifts travel beside them)."""
        return [kvrp.Chunk(k_src=a["srcs"][0], v_src=a["srcs"][1], n_tokens=a["n_tokens"],
                           delta=0 if isinstance(a["delta"], tuple) else a["delta"],
                           k_dst=a["dst"][0], v_dst=a["dst"][1], rank=a["rank"], uk=a["u"][0], vk=a["w"][0],
                           uv=a["u"][1], vv=a["w"][1], src_layer_stride=a["src_layer_stride"],
                           u_layer_stride=a["u_layer_stride"], v_layer_stride=a["w_layer_stride"])
                for a in self._chunks]

    def pools_host(self) -> dict:
        return {n: p.view(torch.int16).cpu().numpy().view(np.uint16) for n, p in self.pools.items()}

    def inputs_host_rows(self, name, layer, rows) -> np.ndarray:
        return self.rows[name][layer, rows].view(torch.int16).cpu().numpy().view(np.uint16)

    def status_value(self) -> int:
        return int(self.status.item())

"""Helpers of the GPU parity tests: run a workload through the C ABI and
compare the destination pools with the fp64 oracle, chunk by chunk."""
from __future__ import annotations

import numpy as np
import torch

import harness
from oracle import chunk_layer_rows, conditioning, operator_rows, placement, row_layout, run_workload
from oracle.compare import parity_report


def merge(a: dict, b: dict) -> dict:
    if not a:
        return dict(b)
    out = {}
    for k in a:
        if k in ("max_ulp",):
            out[k] = max(a[k], b[k])
        elif k.startswith("max_"):
            out[k] = max(a[k], b[k])
        else:
            out[k] = a[k] + b[k]
    return out


def run_and_compare(wl, host=None, device="cuda"):
    """Full comparison of every pool element (small workloads).  Returns
    (report per tensor, got pools, oracle pools, device workload)."""
    dwl = harness.DeviceWorkload(wl, device, host=host)
    dwl.run()
    torch.cuda.synchronize()
    got = dwl.pools_host()
    want, refs, conds = run_workload(wl, dwl.host)
    reports = {}
    for name in wl.tensors:
        untouched = np.isnan(refs[name]).all(axis=-1)
        assert np.array_equal(got[name][untouched], want[name][untouched]), f"{name}: untargeted slots changed"
        reports[name] = parity_report(got[name][~untouched], refs[name][~untouched], conds[name][~untouched])
    return reports, got, want, dwl


def streaming_compare(wl, dwl, got=None, layers=None):
    """Chunk-by-chunk comparison for workloads too big for run_workload; the
    inputs must be host-drawn (dwl.host)."""
    got = dwl.pools_host() if got is None else got
    reports = {n: {} for n in wl.tensors}
    for ci, c in enumerate(wl.chunks):
        pages, slots = placement(wl, c)
        for name in wl.tensors:
            for l in (range(wl.n_layers) if layers is None else layers):
                ref, cond = chunk_layer_rows(wl, dwl.host, ci, name, l)
                g = got[name][l, pages, slots]
                reports[name] = merge(reports[name], parity_report(g, ref, cond))
    return reports


def sampled_compare(wl, dwl, n_rows=48, seed=0):
    """Compare randomly chosen output rows (any workload size): the inputs of
    those rows are copied back from the device and given to the oracle."""
    rng = np.random.default_rng(seed)
    reports = {n: {} for n in wl.tensors}
    for _ in range(n_rows):
        ci = int(rng.integers(len(wl.chunks)))
        c = wl.chunks[ci]
        name = wl.tensors[int(rng.integers(len(wl.tensors)))]
        l = int(rng.integers(wl.n_layers))
        toks = np.unique(rng.integers(0, c.n_tokens, size=4))
        dev = dwl.rows[name].device
        t_idx = torch.as_tensor(toks, device=dev)
        x = bits(dwl.rows[name][l, c.src_row0 + t_idx])
        u = w = None
        if c.rank:
            u = bits(dwl.u[name][ci][l, t_idx])
            w = bits(dwl.w[name][ci][l])
        lay = row_layout(wl.family, name, n_heads=wl.n_heads, head_dim=wl.head_dim,
                         kv_lora_dim=wl.kv_lora_dim, rope_dim=wl.rope_dim)
        sec = wl.mrope_sections
        ref = operator_rows(x, u, w, c.delta, wl.theta, lay, sec)
        cond = conditioning(x, u, w, c.delta, wl.theta, lay, sec)
        q = c.dst_start + toks
        page = wl.block_tables[c.seq][q // 16] if wl.paged else q // 16
        pool = dwl.pools[name]
        g = bits(pool[l, torch.as_tensor(page, device=dev), torch.as_tensor(q % 16, device=dev)])
        reports[name] = merge(reports[name], parity_report(g, ref, cond))
    return reports


def layer_compare(wl, dwl, layer: int):
    """Every element of one whole layer (every chunk, every tensor) against the
    oracle, for workloads of any size: each chunk's inputs of that layer are
    copied back from the device, the oracle evaluates them, and the rows the
    device wrote are gathered through the block table."""
    reports = {n: {} for n in wl.tensors}
    for ci, c in enumerate(wl.chunks):
        dev = dwl.rows[wl.tensors[0]].device
        q = c.dst_start + np.arange(c.n_tokens)
        page = wl.block_tables[c.seq][q // 16] if wl.paged else q // 16
        pg, sl = torch.as_tensor(page, device=dev), torch.as_tensor(q % 16, device=dev)
        for name in wl.tensors:
            x = bits(dwl.rows[name][layer, c.src_row0:c.src_row0 + c.n_tokens])
            u = w = None
            if c.rank:
                u = bits(dwl.u[name][ci][layer])
                w = bits(dwl.w[name][ci][layer])
            lay = row_layout(wl.family, name, n_heads=wl.n_heads, head_dim=wl.head_dim,
                             kv_lora_dim=wl.kv_lora_dim, rope_dim=wl.rope_dim)
            ref = operator_rows(x, u, w, c.delta, wl.theta, lay, wl.mrope_sections)
            cond = conditioning(x, u, w, c.delta, wl.theta, lay, wl.mrope_sections)
            g = bits(dwl.pools[name][layer, pg, sl])
            reports[name] = merge(reports[name], parity_report(g, ref, cond))
    return reports


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

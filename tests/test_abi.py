"""The C ABI without a GPU: the library loads, exports every entry point that
include/kvrp.h declares, and rejects bad arguments with the documented status
codes before touching CUDA."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def kvrp():
    from position_invariant_kv_gb300.build import build
    build()
    import position_invariant_kv_gb300 as m
    m.lib()
    return m


def header_functions():
    text = open(os.path.join(ROOT, "include", "kvrp.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\**\s+\**(\w+)\s*\(", text, flags=re.M)))


def test_exports_every_declared_symbol(kvrp):
    declared = header_functions()
    assert set(declared) == set(kvrp.EXPORTED_SYMBOLS), declared
    lib = C.CDLL(kvrp.lib_path)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version(kvrp):
    assert kvrp.kvrp_status_string(0) == "KVRP_OK"
    assert kvrp.kvrp_status_string(5) == "KVRP_ERR_WORKSPACE"
    assert kvrp.kvrp_version() >= 100


def _dst(**kw):
    d = dict(base=0x10000, num_pages=16, layer_stride=16 * 16 * 256)
    d.update(kw)
    return d


def _call(kvrp, **over):
    args = dict(k_src=0x20000, v_src=0x30000, n_layers=1, n_tokens=100, n_kv_heads=2, head_dim=128,
                delta=5, rope_theta=1e4, rank=0)
    kd = over.pop("k_dst", _dst())
    vd = over.pop("v_dst", _dst(base=0x40000))
    args.update(over)
    k, v = args.pop("k_src"), args.pop("v_src")
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_patch(k, v, k_dst=kvrp.Dst(**kd), v_dst=kvrp.Dst(**vd), stream=0, **args)
    return e.value.status


def test_rejects_bad_arguments_before_cuda(kvrp):
    assert _call(kvrp, k_src=0) == kvrp.KVRP_ERR_INVALID_ARG
    assert _call(kvrp, k_src=0x20008) == kvrp.KVRP_ERR_ALIGNMENT
    assert _call(kvrp, head_dim=96) == kvrp.KVRP_ERR_UNSUPPORTED
    f = dict(uk=0x50000, vk=0x60000, uv=0x70000, vv=0x80000)
    assert _call(kvrp, rank=12, **f) == kvrp.KVRP_ERR_UNSUPPORTED         # not a multiple of 8
    assert _call(kvrp, rank=136, **f) == kvrp.KVRP_ERR_UNSUPPORTED        # above 128
    assert _call(kvrp, rank=8, **f) == kvrp.KVRP_ERR_CUDA                 # accepted; no GPU here
    assert _call(kvrp, rank=16) == kvrp.KVRP_ERR_INVALID_ARG            # factors missing
    assert _call(kvrp, rank=0, uk=0x50000) == kvrp.KVRP_ERR_INVALID_ARG  # factors without rank
    assert _call(kvrp, n_tokens=-1) == kvrp.KVRP_ERR_INVALID_ARG
    assert _call(kvrp, n_layers=0) == kvrp.KVRP_ERR_INVALID_ARG
    assert _call(kvrp, rope_theta=-1.0) == kvrp.KVRP_ERR_INVALID_ARG
    assert _call(kvrp, k_dst=_dst(page_size=32)) == kvrp.KVRP_ERR_UNSUPPORTED
    assert _call(kvrp, k_dst=_dst(num_pages=2)) == kvrp.KVRP_ERR_INVALID_ARG   # contiguous too small
    assert _call(kvrp, k_dst=_dst(dst_start=-3)) == kvrp.KVRP_ERR_INVALID_ARG
    assert _call(kvrp, k_dst=_dst(block_table=0x1002)) == kvrp.KVRP_ERR_ALIGNMENT
    assert _call(kvrp, n_layers=2, src_layer_stride=10) == kvrp.KVRP_ERR_INVALID_ARG
    assert _call(kvrp, n_layers=2, src_layer_stride=100 * 256 + 4) == kvrp.KVRP_ERR_ALIGNMENT


def test_mla_and_batch_argument_checks(kvrp):
    d = kvrp.Dst(base=0x10000, num_pages=16, layer_stride=16 * 16 * 576)
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_patch_mla(0x20000, n_layers=1, n_tokens=10, kv_lora_dim=512, rope_dim=32,
                                   delta=1, rope_theta=1e4, dst=d, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_UNSUPPORTED
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_patch_mla(0x20000, n_layers=1, n_tokens=10, kv_lora_dim=500, rope_dim=64,
                                   delta=1, rope_theta=1e4, dst=d, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_UNSUPPORTED
    ch = kvrp.Chunk(k_src=0x20000, v_src=0x30000, n_tokens=10, delta=3,
                    k_dst=kvrp.Dst(base=0x10000, num_pages=4), v_dst=kvrp.Dst(base=0x40000, num_pages=4))
    ws = kvrp.kv_relocate_batch_workspace_size(2)
    assert ws > 0 and kvrp.kv_relocate_batch_workspace_size(0) == 0
    with pytest.raises(kvrp.KvrpError) as e:   # no workspace
        kvrp.kv_relocate_batch([ch, ch], n_layers=1, n_kv_heads=2, head_dim=128, rope_theta=1e4,
                               workspace=0, workspace_bytes=0, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_WORKSPACE
    with pytest.raises(kvrp.KvrpError) as e:   # workspace too small
        kvrp.kv_relocate_batch([ch, ch], n_layers=1, n_kv_heads=2, head_dim=128, rope_theta=1e4,
                               workspace=0x100000, workspace_bytes=ws - 1, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_WORKSPACE
    bad = kvrp.Chunk(k_src=0x20000, v_src=0, n_tokens=10, delta=3,
                     k_dst=kvrp.Dst(base=0x10000, num_pages=4), v_dst=kvrp.Dst(base=0x40000, num_pages=4))
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_batch([ch, bad], n_layers=1, n_kv_heads=2, head_dim=128, rope_theta=1e4,
                               workspace=0x100000, workspace_bytes=ws, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_INVALID_ARG and "chunk 1" in str(e.value)


def test_mla_and_mrope_batch_argument_checks(kvrp):
    d = kvrp.Dst(base=0x10000, num_pages=16, layer_stride=16 * 16 * 576)
    ws = kvrp.kv_relocate_batch_workspace_size(2)
    ch = kvrp.MlaChunk(src=0x20000, n_tokens=10, delta=-7, dst=d)
    with pytest.raises(kvrp.KvrpError) as e:                    # rope_dim must be 64
        kvrp.kv_relocate_batch_mla([ch, ch], n_layers=1, kv_lora_dim=512, rope_dim=32, rope_theta=1e4,
                                   workspace=0x100000, workspace_bytes=ws, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_UNSUPPORTED
    with pytest.raises(kvrp.KvrpError) as e:                    # workspace too small
        kvrp.kv_relocate_batch_mla([ch, ch], n_layers=1, kv_lora_dim=512, rope_dim=64, rope_theta=1e4,
                                   workspace=0x100000, workspace_bytes=ws - 1, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_WORKSPACE
    bad = kvrp.MlaChunk(src=0x20000, n_tokens=10, delta=-7, dst=d, rank=16)   # rank without factors
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_batch_mla([ch, bad], n_layers=1, kv_lora_dim=512, rope_dim=64, rope_theta=1e4,
                                   workspace=0x100000, workspace_bytes=ws, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_INVALID_ARG and "chunk 1" in str(e.value)
    g = kvrp.Chunk(k_src=0x20000, v_src=0x30000, n_tokens=10, delta=3,
                   k_dst=kvrp.Dst(base=0x10000, num_pages=4), v_dst=kvrp.Dst(base=0x40000, num_pages=4))
    with pytest.raises(kvrp.KvrpError) as e:                    # sections must cover head_dim / 2 pairs
        kvrp.kv_relocate_batch_mrope([g, g], [(1, 2, 3), (4, 5, 6)], n_layers=1, n_kv_heads=2, head_dim=128,
                                     mrope_section=(16, 24, 23), rope_theta=1e6, workspace=0x100000,
                                     workspace_bytes=ws, stream=0)
    assert e.value.status == kvrp.KVRP_ERR_INVALID_ARG
    with pytest.raises(ValueError):                             # one shift triple per chunk
        kvrp.kv_relocate_batch_mrope([g, g], [(1, 2, 3)], n_layers=1, n_kv_heads=2, head_dim=128,
                                     mrope_section=(16, 24, 24), rope_theta=1e6, workspace=0x100000,
                                     workspace_bytes=ws, stream=0)


def test_no_gpu_means_cuda_error_not_fallback(kvrp):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_patch(0x20000, 0x30000, n_layers=1, n_tokens=100, n_kv_heads=2, head_dim=128,
                               delta=5, rope_theta=1e4, k_dst=kvrp.Dst(**_dst()),
                               v_dst=kvrp.Dst(**_dst(base=0x40000)), stream=0)
    assert e.value.status == kvrp.KVRP_ERR_CUDA


def test_mrope_argument_checks(kvrp):
    kd, vd = kvrp.Dst(**_dst()), kvrp.Dst(**_dst(base=0x40000))
    base = dict(n_layers=1, n_tokens=100, n_kv_heads=2, head_dim=128, rope_theta=1e4, k_dst=kd, v_dst=vd, stream=0)
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_patch_mrope(0x20000, 0x30000, delta_thw=(1, 2, 3), mrope_section=(16, 24, 20), **base)
    assert e.value.status == kvrp.KVRP_ERR_INVALID_ARG and "sum" in str(e.value)
    with pytest.raises(kvrp.KvrpError) as e:
        kvrp.kv_relocate_patch_mrope(0x20000, 0x30000, delta_thw=(1, 2, 3), mrope_section=(-1, 33, 32), **base)
    assert e.value.status == kvrp.KVRP_ERR_INVALID_ARG
    with pytest.raises(kvrp.KvrpError) as e:     # well-formed: fails only for want of a GPU
        kvrp.kv_relocate_patch_mrope(0x20000, 0x30000, delta_thw=(1, 2, 3), mrope_section=(16, 24, 24), **base)
    import torch
    assert e.value.status == (kvrp.KVRP_ERR_CUDA if not torch.cuda.is_available() else e.value.status)


def test_patch_form_argument_checks(kvrp):
    def status(**over):
        args = dict(conditioned=0x20000, canonical=0x30000, n_layers=2, n_tokens=100, row_width=256,
                    rope_kind=kvrp.KVRP_ROPE_HEADS, rot_dim=128, delta=5, rope_theta=1e4, rank=16, oversample=8,
                    power_iters=2, omega=0x50000, u_out=0x60000, v_out=0x70000, workspace=0x100000,
                    workspace_bytes=1 << 30, cond_layer_stride=100 * 256, canon_layer_stride=100 * 256,
                    u_layer_stride=100 * 16, v_layer_stride=256 * 16, stream=0)
        args.update(over)
        c, x = args.pop("conditioned"), args.pop("canonical")
        with pytest.raises(kvrp.KvrpError) as e:
            kvrp.kv_patch_form(c, x, **args)
        return e.value.status

    assert status(conditioned=0) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(omega=0x50004) == kvrp.KVRP_ERR_ALIGNMENT
    assert status(rank=64, oversample=40) == kvrp.KVRP_ERR_UNSUPPORTED      # rank + oversample > 96
    assert status(rank=0) == kvrp.KVRP_ERR_UNSUPPORTED
    assert status(rot_dim=96) == kvrp.KVRP_ERR_INVALID_ARG                   # 256 is not a multiple of 96
    assert status(rot_dim=130) == kvrp.KVRP_ERR_UNSUPPORTED
    assert status(rope_kind=7) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(rope_kind=kvrp.KVRP_ROPE_MLA_TAIL, row_width=64, rot_dim=64) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(power_iters=9) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(cond_layer_stride=10) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(v_layer_stride=10) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(workspace_bytes=1024) == kvrp.KVRP_ERR_WORKSPACE
    need = kvrp.kv_patch_form_workspace_size(2, 100, 256, 16, 8)
    assert need >= 4 * 2 * 100 * 256                                          # at least the fp32 deficit
    assert kvrp.kv_patch_form_workspace_size(0, 100, 256, 16, 8) == 0
    import torch
    if not torch.cuda.is_available():                                         # well-formed: no GPU, no fallback
        assert status(workspace_bytes=need) == kvrp.KVRP_ERR_CUDA


def test_patch_form_orbit_argument_checks(kvrp):
    def status(conds, deltas, **over):
        args = dict(n_layers=1, n_tokens=100, row_width=256, rope_kind=kvrp.KVRP_ROPE_HEADS, rot_dim=128,
                    rope_theta=1e4, rank=16, oversample=8, power_iters=1, omega=0x50000, u_out=0x60000,
                    v_out=0x70000, workspace=0x100000, workspace_bytes=1 << 30, stream=0)
        args.update(over)
        with pytest.raises(kvrp.KvrpError) as e:
            kvrp.kv_patch_form_orbit(conds, deltas, 0x30000, **args)
        return e.value.status

    assert status([], []) == kvrp.KVRP_ERR_UNSUPPORTED
    assert status([0x20000] * 65, list(range(65))) == kvrp.KVRP_ERR_UNSUPPORTED
    assert status([0x20000, 0], [1, 2]) == kvrp.KVRP_ERR_INVALID_ARG
    assert status([0x20000, 0x20008], [1, 2]) == kvrp.KVRP_ERR_ALIGNMENT
    assert status([0x20000], [1], row_width=254, rope_kind=kvrp.KVRP_ROPE_NONE) == kvrp.KVRP_ERR_UNSUPPORTED
    with pytest.raises(ValueError):
        kvrp.kv_patch_form_orbit([0x20000], [1, 2], 0x30000, n_layers=1, n_tokens=100, row_width=256,
                                 rope_kind=0, rot_dim=0, rope_theta=1e4, rank=16, oversample=8, power_iters=1,
                                 omega=0x50000, u_out=0x60000, v_out=0x70000, workspace=0x100000)


def test_attend_argument_checks(kvrp):
    """kv_attend_relocated validates everything on the host, before any CUDA call."""
    def chunk(**over):
        c = dict(k=0x20000, v=0x30000, n_tokens=100, delta=5, rank=16, uk=0x40000, vk=0x50000, uv=0x60000,
                 vv=0x70000)
        c.update(over)
        return kvrp.AttnChunk(**c)

    def status(chunks=None, seq_chunks=None, q=0x80000, **over):
        args = dict(n_q_heads=8, n_kv_heads=2, head_dim=128, rope_theta=1e6, softmax_scale=0.088, out=0x90000,
                    workspace=0x100000, workspace_bytes=1 << 40, stream=0)
        args.update(over)
        chunks = [chunk()] if chunks is None else chunks
        seq_chunks = [0, len(chunks)] if seq_chunks is None else seq_chunks
        with pytest.raises(kvrp.KvrpError) as e:
            kvrp.kv_attend_relocated(q, chunks, seq_chunks, **args)
        return e.value.status

    assert status(q=0) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(q=0x80004) == kvrp.KVRP_ERR_ALIGNMENT
    assert status(head_dim=96) == kvrp.KVRP_ERR_UNSUPPORTED
    assert status(n_q_heads=7) == kvrp.KVRP_ERR_UNSUPPORTED                  # not a multiple of n_kv_heads
    assert status(n_q_heads=64) == kvrp.KVRP_ERR_UNSUPPORTED                 # 32 query heads per KV head
    assert status(rope_theta=0.0) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(softmax_scale=-1.0) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(chunks=[chunk(rank=24)]) == kvrp.KVRP_ERR_UNSUPPORTED      # rank not a multiple of 16
    assert status(chunks=[chunk(rank=144)]) == kvrp.KVRP_ERR_UNSUPPORTED
    assert status(chunks=[chunk(uk=None)]) == kvrp.KVRP_ERR_INVALID_ARG      # rank > 0 needs all four factors
    assert status(chunks=[chunk(n_tokens=-1)]) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(chunks=[chunk(k=None)]) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(chunks=[chunk(k=0x20008)]) == kvrp.KVRP_ERR_ALIGNMENT
    assert status(chunks=[chunk(vv=0x70004)]) == kvrp.KVRP_ERR_ALIGNMENT
    assert status(chunks=[chunk(block_table=0x1000, num_pages=0)]) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(chunks=[chunk(block_table=0x1002, num_pages=4)]) == kvrp.KVRP_ERR_ALIGNMENT
    assert status(seq_chunks=[0, 0]) == kvrp.KVRP_ERR_INVALID_ARG            # must end at n_chunks
    assert status(chunks=[chunk(), chunk()], seq_chunks=[0, 2, 1, 2]) == kvrp.KVRP_ERR_INVALID_ARG
    assert status(chunks=[chunk()] * 257, seq_chunks=[0, 257]) == kvrp.KVRP_ERR_UNSUPPORTED
    assert status(workspace_bytes=16) == kvrp.KVRP_ERR_WORKSPACE
    need = kvrp.kv_attend_relocated_workspace_size([100], 8, 2, 128)
    assert need > 0
    assert kvrp.kv_attend_relocated_workspace_size([], 8, 2, 128) == 0
    assert kvrp.kv_attend_relocated_workspace_size([100], 8, 3, 128) == 0     # heads not a multiple
    import torch
    if not torch.cuda.is_available():                                         # well-formed: no GPU, no fallback
        assert status(workspace_bytes=need) == kvrp.KVRP_ERR_CUDA
        assert status(workspace_bytes=need, chunks=[chunk(block_table=0x1000, num_pages=7)]) == kvrp.KVRP_ERR_CUDA

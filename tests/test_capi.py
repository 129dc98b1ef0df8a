"""The C-ABI library builds, loads and exports every symbol include/moestep.h declares;
host-side validation rejects bad arguments before any CUDA call (no GPU needed)."""
import ctypes
import os
import re

import pytest

from moe_decode_step_router_gb300 import build as mbuild
from moe_decode_step_router_gb300 import moestep as ms
from moe_decode_step_router_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    mbuild.build()
    return ms.lib()


def _declared():
    src = open(os.path.join(ROOT, "include", "moestep.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 17
    assert set(names) == set(ms.EXPORTS)
    for n in names:
        assert getattr(lib, n) is not None


def _desc(name="tiny_mxfp8", **over):
    return ms.layer_desc(synth.config(name, **over), synth.act_global_scales(synth.config(name, **over)))


def test_sizes(lib):
    d = _desc()
    # W13: 2I/128 blocks * H/128 steps * (16 KiB + one 512-byte scale atom) per expert
    assert ms.moe_packed_bytes(d, ms.MOE_W13) == 16 * (512 // 128) * (1024 // 128) * (16384 + 512)
    assert ms.moe_packed_bytes(d, ms.MOE_W2) == 16 * (1024 // 128) * (256 // 128) * (16384 + 512)
    assert ms.moe_packed_bytes(d, ms.MOE_SH13) == 1 * 4 * 8 * (16384 + 512)
    assert ms.moe_act_bytes(ms.MOE_FMT_MXFP8, 5, 1024) == 16 * 1024
    assert ms.moe_act_scale_bytes(ms.MOE_FMT_NVFP4, 5, 1024) == (512 // 128) * 4 * 512
    assert ms.moe_workspace_bytes(d) > 0
    nv = _desc("nvfp4_h4096_e512_k10")
    assert ms.moe_packed_bytes(nv, ms.MOE_W13) == 512 * (2048 // 128) * (2048 // 128) * (16384 + 2048)


@pytest.mark.parametrize("field,value,status", [
    ("H", 1000, ms.MOE_ERR_INVALID_ARG), ("E", 0, ms.MOE_ERR_INVALID_ARG), ("k", 17, ms.MOE_ERR_INVALID_ARG),
    ("I", 300, ms.MOE_ERR_INVALID_ARG), ("w_fmt", ms.MOE_FMT_BF16, ms.MOE_ERR_UNSUPPORTED),
    ("shared_fmt", 7, ms.MOE_ERR_UNSUPPORTED), ("swiglu_limit", float("nan"), ms.MOE_ERR_INVALID_ARG),
    ("gemm_schedule", 3, ms.MOE_ERR_INVALID_ARG), ("gemm_schedule", -1, ms.MOE_ERR_INVALID_ARG),
    ("ffn_launches", 3, ms.MOE_ERR_INVALID_ARG), ("front_launches", -1, ms.MOE_ERR_INVALID_ARG)])
def test_bad_descriptor_rejected(lib, field, value, status):
    d = _desc()
    setattr(d, field, value)
    assert ms.moe_workspace_bytes(d) == 0
    st = lib.moe_workspace_init(ctypes.byref(d), ctypes.c_void_p(1 << 20), None)
    assert st == status
    assert lib.moe_last_error_string().decode() != ""


def test_bad_rows_and_pointers_rejected_before_launch(lib):
    d = _desc()
    fake = 1 << 20  # never dereferenced: validation fails first
    st = lib.moe_router_topk(ctypes.byref(d), fake, fake, None, None, 0, None, fake, fake, fake, fake, None, None,
                             fake, None)
    assert st == ms.MOE_ERR_INVALID_ARG and "M=0" in lib.moe_last_error_string().decode()
    st = lib.moe_router_topk(ctypes.byref(d), fake + 8, fake, None, None, 1, None, fake, fake, fake, fake, None,
                             None, fake, None)
    assert st == ms.MOE_ERR_INVALID_ARG and "aligned" in lib.moe_last_error_string().decode()
    st = lib.moe_route_tiles(ctypes.byref(d), fake, 65, fake, fake, fake, fake, fake, fake, None)
    assert st == ms.MOE_ERR_INVALID_ARG
    args = ms.StepArgs()
    st = lib.moe_step(ctypes.byref(d), ctypes.byref(args), 1, fake, None)
    assert st == ms.MOE_ERR_INVALID_ARG and "NULL" in lib.moe_last_error_string().decode()
    nv = _desc("nvfp4_h6144_e256_k8_16rows")
    q = ms.QWeight(fake, None)  # NVFP4 needs global scales
    st = lib.moe_expert_gate_up(ctypes.byref(nv), ctypes.byref(q), ctypes.byref(q), fake, fake, fake, None, fake, 4,
                                fake, fake, fake, None)
    assert st == ms.MOE_ERR_INVALID_ARG and "global_scale" in lib.moe_last_error_string().decode()
    st = lib.moe_expert_ffn(ctypes.byref(nv), ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                            fake, fake, fake, None, fake, 4, fake, fake, fake, fake, None)
    assert st == ms.MOE_ERR_INVALID_ARG and "global_scale" in lib.moe_last_error_string().decode()
    st = lib.moe_expert_ffn(ctypes.byref(d), ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), ctypes.byref(q),
                            fake, fake, fake, None, fake, 4, fake, fake, None, fake, None)
    assert st == ms.MOE_ERR_INVALID_ARG and "y_pairs" in lib.moe_last_error_string().decode()
    with pytest.raises(ms.MoeError):
        ms._check(ms.MOE_ERR_INVALID_ARG)


# Every region moe_ws_view hands out, at the largest step (64 rows), with its size from
# the shapes the header documents: inside the workspace, 16-byte aligned, and disjoint
# from every other region (the shared FC1 input may alias the routed one when the
# formats agree). Host arithmetic only: the base address is never dereferenced.
@pytest.mark.parametrize("name", list(synth.CONFIGS) + ["nv_bf16_shared"])
def test_workspace_regions_are_disjoint_and_aligned(lib, name):
    cfg = (synth.config("nvfp4_h6144_e256_k8_16rows", H=1024, E=16, k=4, I=256, I_sh=256) if name == "nv_bf16_shared"
           else synth.config(name))
    d = ms.layer_desc(cfg, synth.act_global_scales(cfg))
    total = ms.moe_workspace_bytes(d)
    base = 1 << 40
    v = ms.WsPtrs()
    assert lib.moe_ws_view(ctypes.byref(d), ctypes.c_void_p(base), ctypes.byref(v)) == 0
    M, E, k, H = 64, cfg["E"], cfg["k"], cfg["H"]
    P = M * k + M
    fr, fs = cfg["w_fmt"], cfg["sh_fmt"]
    size = {
        "status": 32, "logits": 4 * M * E, "scores": 4 * M * E, "topk_idx": 4 * M * k, "topk_w": 4 * M * k,
        "expert_counts": 4 * (E + 1), "perm": 4 * P, "inv_perm": 4 * P, "tiles": 12 * (P + E + 1), "num_tiles": 4,
        "xq": ms.moe_act_bytes(fr, M, H), "xq_scales": ms.moe_act_scale_bytes(fr, M, H),
        "xq_shared": ms.moe_act_bytes(fs, M, H), "xq_shared_scales": ms.moe_act_scale_bytes(fs, M, H),
        "hq": ms.moe_hq_bytes(d, M), "hq_scales": ms.moe_hq_scale_bytes(d, M), "y_pairs": 4 * P * H}
    regions = []
    for field, n in size.items():
        ptr = getattr(v, field)
        assert ptr is not None and ptr % 16 == 0, field
        assert base <= ptr and ptr + n <= base + total, field
        if n:
            regions.append((ptr, ptr + n, field))
    regions.sort()
    for (a0, a1, fa), (b0, b1, fb) in zip(regions, regions[1:]):
        if a0 == b0 and {fa, fb} in ({"xq", "xq_shared"}, {"xq_scales", "xq_shared_scales"}) and fr == fs:
            continue  # the routed and shared FC1 inputs are one buffer when the formats agree
        assert a1 <= b0, "%s overlaps %s" % (fa, fb)


def test_workspace_size_follows_the_schedule(lib):
    """The counter-fed schedules need the pool's partial-sum slots (4 per CTA of 64 x 128
    fp32); the default static schedule does not carry them."""
    cfg = synth.config("mxfp8_h7168_e256_k8_8rows")
    sizes = {}
    for name in ("static", "hybrid", "dynamic"):
        d = ms.layer_desc(dict(cfg, schedule=name), synth.act_global_scales(cfg))
        sizes[name] = ms.moe_workspace_bytes(d)
    slot = 64 * 128 * 4
    assert sizes["hybrid"] == sizes["dynamic"]
    assert sizes["hybrid"] - sizes["static"] == (4 * 160 - 2 * 160) * slot
    d = ms.layer_desc(dict(cfg, ffn_launches=2), synth.act_global_scales(cfg))
    assert ms.moe_workspace_bytes(d) == sizes["static"]

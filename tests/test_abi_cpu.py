"""The C ABI library builds, loads and exports every declared entry point;
pure entry points and argument validation work without a GPU."""

import ctypes
import os
import re

import pytest

from host_paged_expert_gb300 import _lib, synth
from host_paged_expert_gb300.synth import MoEShape

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "pe.h")


@pytest.fixture(scope="module")
def L():
    if not os.path.exists(_lib.LIB_PATH):
        from host_paged_expert_gb300 import build

        build.build()
    return _lib.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(pe_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("pe_create", "pe_load_host_expert", "pe_forward", "pe_stats", "pe_destroy",
                 "pe_last_error", "pe_required_device_bytes", "pe_reset_residency"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), f"{n} declared in pe.h but not exported"
    assert sorted(_lib.EXPORTS) == names


def test_row_layout_matches_expert_sizes(L):
    bf = _lib.row_layout(synth.STACK48)
    assert bf["payload_bytes"] == 9_437_184 == synth.STACK48.expert_bytes
    assert bf["row_stride"] == 9_437_184
    assert bf["w2_offset"] == 6_291_456
    f8 = _lib.row_layout(synth.STACK48_FP8)
    assert f8["payload_bytes"] == 4_719_744 == synth.STACK48_FP8.expert_bytes
    assert f8["s13_bytes"] == 4 * 12 * 16 and f8["s2_bytes"] == 4 * 16 * 6
    for k in ("w13_offset", "s13_offset", "w2_offset", "s2_offset"):
        assert f8[k] % 128 == 0
    assert f8["row_stride"] % 256 == 0 and f8["row_stride"] >= f8["s2_offset"] + f8["s2_bytes"]
    tiny = _lib.row_layout(synth.TINY)
    assert tiny["payload_bytes"] == 3 * 256 * 128 * 2
    i4 = _lib.row_layout(synth.STACK48_INT4)  # the pages' 2.43 MB GPTQ int4 expert
    assert i4["payload_bytes"] == 2_433_024 == synth.STACK48_INT4.expert_bytes
    assert i4["w13_bytes"] == 1536 * 1024 and i4["w2_bytes"] == 2048 * 384
    assert i4["s13_bytes"] == 2 * 1536 * 16 and i4["s2_bytes"] == 2 * 2048 * 6
    for k in ("w13_offset", "s13_offset", "w2_offset", "s2_offset"):
        assert i4[k] % 128 == 0


def test_fp4_row_layouts(L):
    """MXFP4: codes plus one E8M0 byte per 32 inputs; NVFP4: one E4M3 byte
    per 16 inputs plus a 16-byte tensor-scale header per grid.  An
    intermediate width that is not a multiple of 128 is carried padded to the
    next multiple (2880 -> 2944), in codes and scales alike."""
    H, I = 2048, 768
    mx = _lib.row_layout(synth.STACK48_MXFP4)
    assert mx["w13_bytes"] == 2 * I * H // 2 and mx["w2_bytes"] == H * I // 2
    assert mx["s13_bytes"] == 2 * I * H // 32 and mx["s2_bytes"] == H * I // 32
    assert mx["payload_bytes"] == synth.STACK48_MXFP4.expert_bytes == 2_506_752
    nv = _lib.row_layout(synth.STACK48_NVFP4)
    assert nv["s13_bytes"] == 16 + 2 * I * H // 16 and nv["s2_bytes"] == 16 + H * I // 16
    assert nv["payload_bytes"] == synth.STACK48_NVFP4.expert_bytes + 2 * 12  # headers pad the two fp32 scales
    for k in ("w13_offset", "s13_offset", "w2_offset", "s2_offset"):
        assert mx[k] % 128 == 0 and nv[k] % 128 == 0
    pad = _lib.row_layout(synth.MoEShape(1, 8, 2, 3, 256, 2880, "mxfp4"))
    assert pad["w13_bytes"] == 2 * 2944 * 256 // 2 and pad["w2_bytes"] == 256 * 2944 // 2
    assert pad["s13_bytes"] == 2 * 2944 * 256 // 32 and pad["s2_bytes"] == 256 * 2944 // 32


@pytest.mark.parametrize("dtype,H,I", [("mxfp4", 200, 256), ("mxfp4", 256, 48), ("nvfp4", 256, 40)])
def test_fp4_shape_rules(L, dtype, H, I):
    """H must be a multiple of 128; I a multiple of the format's block."""
    cfg = _lib.make_config(synth.MoEShape(1, 8, 2, 4, H, I, dtype), 4, 0)
    assert L.pe_required_device_bytes(ctypes.byref(cfg)) == 0


def test_external_store_argument_checks(L):
    """pe_create_external refuses a NULL, misaligned or too small host store
    before it touches the device."""
    import numpy as np

    cfg = _lib.make_config(synth.TINY, 4)
    need = _lib.host_store_bytes(synth.TINY)
    buf = np.zeros(need + 8192, np.uint8)
    base = (buf.ctypes.data + 4095) // 4096 * 4096
    h = ctypes.c_void_p()
    for ptr, n in ((None, need), (base + 8, need), (base, need - 1)):
        st = L.pe_create_external(ctypes.byref(cfg), None, 0, ptr, n, 1, ctypes.byref(h))
        assert st == _lib.PE_ERR_INVALID, (ptr, n)
        assert b"external host store" in L.pe_last_error(None)


def test_max_waves_from_shapes(L):
    s = synth.STACK48
    assert _lib.max_waves(s, 1) == 1
    assert _lib.max_waves(s, 4) == 1           # 32 entries fit K=32
    assert _lib.max_waves(s, 5) == 2           # 40 entries, 40 distinct at most
    assert _lib.max_waves(s, 2048) == 4        # at most E=128 distinct
    assert _lib.max_waves(s.with_slots(128), 2048) == 1
    assert _lib.max_waves(synth.TINY, 64) == 3  # 16 experts over K=6


def test_required_bytes_cover_slot_table(L):
    s = synth.STACK48
    n = _lib.required_device_bytes(s, 8)
    table = s.num_layers * s.num_slots * 9_437_184
    assert table <= n < table + 64 * 2**20
    assert _lib.required_device_bytes(s.with_slots(64), 8) > n


@pytest.mark.parametrize("bad", [
    dict(num_slots=1),            # K < top_k
    dict(num_slots=200),          # K > E
    dict(top_k=0),
    dict(hidden=100),             # not a multiple of 8
    dict(num_experts=2000),
])
def test_invalid_configs_rejected(L, bad):
    base = dict(num_layers=2, num_experts=16, top_k=2, num_slots=6, hidden=256, intermediate=128)
    base.update(bad)
    s = MoEShape(**base)
    cfg = _lib.make_config(s, 4)
    assert L.pe_required_device_bytes(ctypes.byref(cfg)) == 0
    h = ctypes.c_void_p()
    st = L.pe_create(ctypes.byref(cfg), None, 0, ctypes.byref(h))
    assert st == _lib.PE_ERR_INVALID
    assert L.pe_last_error(None)


def test_unsupported_dtype_and_fp8_shape(L):
    cfg = _lib.make_config(synth.TINY, 4)
    cfg.dtype = 7
    h = ctypes.c_void_p()
    assert L.pe_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == _lib.PE_ERR_UNSUPPORTED_DTYPE
    s = MoEShape(1, 16, 2, 6, 200, 128, "fp8")  # H not a multiple of 128
    cfg = _lib.make_config(s, 4)
    assert L.pe_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == _lib.PE_ERR_INVALID
    s = MoEShape(1, 16, 2, 6, 256, 192, "int4")  # I not a multiple of the 128-input group
    cfg = _lib.make_config(s, 4)
    assert L.pe_create(ctypes.byref(cfg), None, 0, ctypes.byref(h)) == _lib.PE_ERR_INVALID


def test_null_handle_calls_are_errors(L):
    assert L.pe_forward(None, 0, None, None, None, 1, None) == _lib.PE_ERR_INVALID
    assert L.pe_stats(None, -1, None) == _lib.PE_ERR_INVALID
    assert L.pe_load_host_expert(None, 0, 0, None, None, None, None) == _lib.PE_ERR_INVALID
    L.pe_destroy(None)


def test_slots_for_budget(L):
    """The library's K for a budget is the largest K whose whole arena fits,
    and agrees within one slot with the oracle's floor formula (the arena's
    small per-K plan buffers are the difference)."""
    from oracle import sizing

    s = synth.STACK48
    T = 8
    per_slot = s.num_layers * _lib.row_layout(s)["row_stride"]
    need = {K: _lib.required_device_bytes(s.with_slots(K), T) for K in (8, 39, 40, 41, 128)}
    assert _lib.slots_for_budget(s, T, need[40]) == 40
    assert _lib.slots_for_budget(s, T, need[40] - 1) == 39
    assert _lib.slots_for_budget(s, T, need[41] - 1) == 40
    assert _lib.slots_for_budget(s, T, need[128] + 10**9) == 128
    assert _lib.slots_for_budget(s, T, need[8] - 1) == 0
    fixed = need[8] - 8 * per_slot
    for budget in (need[8], 100e9, 200e9, 271e9, need[128] - 1):
        k = _lib.slots_for_budget(s, T, int(budget))
        assert _lib.required_device_bytes(s.with_slots(k), T) <= budget
        if k < s.num_experts:
            assert _lib.required_device_bytes(s.with_slots(k + 1), T) > budget
        assert abs(k - sizing.slots_for_budget(budget, fixed, per_slot, s.num_experts, s.top_k)) <= 1


def test_prefill_arena_holds_one_staging_row_per_slot(L):
    """With the tensor-core prefill path and steps of two or more waves, the
    arena adds K staging rows after the slot table: one slot more costs one
    expert row per layer plus one staging row, against one row per layer at
    decode sizes (the other per-slot buffers are a few hundred bytes)."""
    s = synth.STACK48
    stride = _lib.row_layout(s)["row_stride"]
    assert _lib.max_waves(s, 2048) >= 2
    per_slot_prefill = _lib.required_device_bytes(s, 2048) - _lib.required_device_bytes(s.with_slots(31), 2048)
    per_slot_decode = _lib.required_device_bytes(s, 8) - _lib.required_device_bytes(s.with_slots(31), 8)
    assert abs(per_slot_decode - s.num_layers * stride) < 64 * 1024
    assert abs(per_slot_prefill - per_slot_decode - stride) < 64 * 1024
    # one wave at most (K = E): no staging rows, so the arena beyond the slot
    # table is K rows smaller than at K = 32
    full = s.with_slots(s.num_experts)
    assert _lib.max_waves(full, 2048) == 1
    beyond_full = _lib.required_device_bytes(full, 2048) - s.num_layers * s.num_experts * stride
    beyond_32 = _lib.required_device_bytes(s, 2048) - s.num_layers * s.num_slots * stride
    assert abs(beyond_32 - beyond_full - s.num_slots * stride) < 256 * 1024

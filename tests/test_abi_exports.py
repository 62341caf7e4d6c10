"""The C-ABI library builds, loads and exports every entry point that
include/aq.h declares; host-side validation and size queries work without a
GPU (CPU only: no compute call reaches a device)."""
import ctypes as C
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def aq():
    from nvfp4_block_scaled_aq_gb300 import build
    build.build()
    import nvfp4_block_scaled_aq_gb300.aq as aqmod
    aqmod.lib()
    return aqmod


def declared_symbols():
    text = open(os.path.join(ROOT, "include", "aq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(aq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_symbols()
    for required in ("aq_reconstruct", "aq_quantize_nvfp4", "aq_gemv_nvfp4",
                     "aq_decode_step_weights", "aq_reconstruct_quantize_nvfp4",
                     "aq_poll_device_status", "aq_last_error"):
        assert required in names


def test_every_declared_symbol_is_exported(aq):
    out = subprocess.run(["nm", "-D", "--defined-only", aq.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (aq_[a-z0-9_]+)$", out, flags=re.M))
    missing = [s for s in declared_symbols() if s not in exported]
    assert not missing, missing
    for s in declared_symbols():
        assert hasattr(aq.lib(), s)


def test_exports_are_plain_c(aq):
    out = subprocess.run(["nm", "-D", "--defined-only", aq.LIB_PATH],
                         capture_output=True, text=True, check=True).stdout
    # nothing C++-mangled is exported under the aq_ prefix
    assert not re.search(r"\b_Z\w*aq_", out)


def test_size_queries_match_the_layout_definition(aq, oracle_mod):
    for n, k in ((1536, 1152), (37, 96), (1, 32), (43008, 5376), (5376, 21504)):
        assert aq.packed_bytes(n, k) == n * k // 2
        assert aq.scale_bytes(n, k) == oracle_mod.scale_layout_bytes(n, k)
    for n, k in ((0, 32), (16, 16), (16, 48), (16, 0), (-1, 64)):
        assert aq.packed_bytes(n, k) == 0 and aq.scale_bytes(n, k) == 0
    assert aq.quantize_workspace_bytes() >= 4
    assert aq.lib().aq_version() >= 100


def test_host_validation_without_a_device(aq):
    L = aq.lib()
    bad_k = aq.Nvfp4WeightC(16, 100, 16, 16, 16)
    assert L.aq_gemv_nvfp4(C.byref(bad_k), C.c_void_p(16), 1, C.c_void_p(16), 0,
                           None, 0, None) == aq.ERR_SHAPE
    assert "multiple of 32" in aq.last_error()
    null_w = aq.Nvfp4WeightC(16, 64, None, None, None)
    assert L.aq_gemv_nvfp4(C.byref(null_w), None, 1, None, 0, None, 0, None) == \
        aq.ERR_INVALID_ARG
    misaligned = aq.Nvfp4WeightC(16, 64, 8, 16, 16)
    assert L.aq_gemv_nvfp4(C.byref(misaligned), C.c_void_p(16), 1, C.c_void_p(16), 0,
                           None, 0, None) == aq.ERR_ALIGNMENT
    ok_w = aq.Nvfp4WeightC(16, 64, 256, 256, 256)
    assert L.aq_gemv_nvfp4(C.byref(ok_w), C.c_void_p(16), 0, C.c_void_p(16), 0,
                           None, 0, None) == aq.ERR_SHAPE
    # the GEMV paths take up to AQ_MAX_M tokens, the MMA path (and AUTO) up to
    # AQ_MAX_M_MMA
    assert L.aq_gemv_nvfp4(C.byref(ok_w), C.c_void_p(16), 17, C.c_void_p(16), aq.PATH_GEMV,
                           None, 0, None) == aq.ERR_SHAPE
    assert L.aq_gemv_nvfp4(C.byref(ok_w), C.c_void_p(16), 65, C.c_void_p(16), aq.PATH_AUTO,
                           None, 0, None) == aq.ERR_SHAPE
    assert L.aq_gemv_nvfp4(C.byref(ok_w), C.c_void_p(16), 65, C.c_void_p(16), aq.PATH_MMA,
                           None, 0, None) == aq.ERR_SHAPE
    assert L.aq_quantize_act_nvfp4(C.c_void_p(16), 0, 64, C.c_void_p(16), C.c_void_p(16),
                                   C.c_void_p(16), None) == aq.ERR_SHAPE
    assert L.aq_quantize_act_nvfp4(C.c_void_p(16), 2, 48, C.c_void_p(16), C.c_void_p(16),
                                   C.c_void_p(16), None) == aq.ERR_SHAPE
    assert L.aq_quantize_act_nvfp4(C.c_void_p(8), 2, 64, C.c_void_p(16), C.c_void_p(16),
                                   C.c_void_p(16), None) == aq.ERR_ALIGNMENT
    assert L.aq_gemv_nvfp4(C.byref(ok_w), C.c_void_p(16), 1, C.c_void_p(16), 7,
                           None, 0, None) == aq.ERR_INVALID_ARG
    assert L.aq_reconstruct(None, None, None, None, 16, 64, 0, None, None) == \
        aq.ERR_INVALID_ARG
    assert L.aq_reconstruct(C.c_void_p(16), C.c_void_p(16), None, None, 16, 64, 65,
                            C.c_void_p(16), None) == aq.ERR_SHAPE
    assert L.aq_decode_step_weights(None, -1, None, None, 1, 0, None, 0, None) == \
        aq.ERR_INVALID_ARG
    assert L.aq_decode_step_weights(None, 0, None, None, 1, 0, None, 0, None) == aq.OK
    assert L.aq_quantize_nvfp4(None, 16, 64, None, None, 0, None) == aq.ERR_INVALID_ARG
    # bf16 GEMV: k a multiple of 8, 1 <= m <= AQ_MAX_M, known flags, 16-byte
    # aligned non-NULL buffers -- all checked before any device query
    p16 = C.c_void_p(256)
    assert L.aq_gemv_bf16(p16, 16, 12, p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert L.aq_gemv_bf16(p16, 0, 64, p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert L.aq_gemv_bf16(p16, 16, 64, p16, 0, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert L.aq_gemv_bf16(p16, 16, 64, p16, 17, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert L.aq_gemv_bf16(p16, 16, 64, p16, 1, p16, 2, None, 0, None) == aq.ERR_INVALID_ARG
    assert L.aq_gemv_bf16(None, 16, 64, p16, 1, p16, 0, None, 0, None) == aq.ERR_INVALID_ARG
    assert L.aq_gemv_bf16(C.c_void_p(8), 16, 64, p16, 1, p16, 0, None, 0, None) == \
        aq.ERR_ALIGNMENT
    # runtime low-rank GEMV: rank, s, U/V and flags checked on the host
    lr = L.aq_gemv_lowrank_nvfp4
    assert lr(C.byref(ok_w), p16, p16, p16, 17, p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert lr(C.byref(ok_w), None, None, None, 0, p16, 1, p16, 0, None, 0, None) == \
        aq.ERR_INVALID_ARG
    assert lr(C.byref(ok_w), p16, None, p16, 4, p16, 1, p16, 0, None, 0, None) == \
        aq.ERR_INVALID_ARG
    assert lr(C.byref(ok_w), C.c_void_p(258), p16, p16, 4, p16, 1, p16, 0, None, 0, None) == \
        aq.ERR_ALIGNMENT
    assert lr(C.byref(ok_w), p16, p16, p16, 4, p16, 1, p16, 4, None, 0, None) == \
        aq.ERR_INVALID_ARG
    assert lr(C.byref(ok_w), p16, p16, p16, 4, p16, 17, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert L.aq_gemv_lowrank_workspace_bytes(16, 64, 1, 17) == 0
    # fused gate+up activation: n a multiple of 16, interleave shape checks
    w24 = aq.Nvfp4WeightC(24, 64, 256, 256, 256)
    assert L.aq_gemv_glu_nvfp4(C.byref(w24), p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert L.aq_gemv_glu_nvfp4(C.byref(ok_w), p16, 1, p16, 2, None, 0, None) == aq.ERR_INVALID_ARG
    assert L.aq_interleave_gate_up(p16, 12, 64, p16, None) == aq.ERR_SHAPE
    assert L.aq_interleave_gate_up(p16, 16, 60, p16, None) == aq.ERR_SHAPE
    assert L.aq_interleave_gate_up(None, 16, 64, p16, None) == aq.ERR_INVALID_ARG
    assert L.aq_interleave_gate_up(C.c_void_p(8), 16, 64, p16, None) == aq.ERR_ALIGNMENT
    # per-segment scales: the segment table is checked on the host
    def segs(*e):
        return (C.c_int32 * len(e))(*e)
    w64 = aq.Nvfp4WeightC(64, 64, 256, 256, 256)
    gs = L.aq_gemv_nvfp4_segments
    assert gs(C.byref(w64), 0, segs(64), p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert gs(C.byref(w64), 9, segs(*range(8, 72, 8)), p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert gs(C.byref(w64), 2, segs(40, 30), p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert gs(C.byref(w64), 2, segs(40, 64), p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert gs(C.byref(w64), 2, segs(32, 60), p16, 1, p16, 0, None, 0, None) == aq.ERR_SHAPE
    assert gs(C.byref(w64), 1, None, p16, 1, p16, 0, None, 0, None) == aq.ERR_INVALID_ARG
    assert L.aq_quantize_nvfp4_segments(p16, 64, 64, 2, segs(40, 64), C.byref(w64), None, 0,
                                        None) == aq.ERR_SHAPE
    assert L.aq_gemv_bf16_workspace_bytes(16, 12, 1) == 0
    assert L.aq_gemv_bf16_workspace_bytes(16, 64, 17) == 0


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    import nvfp4_block_scaled_aq_gb300.aq as aqmod
    monkeypatch.setattr(aqmod, "_lib", None)
    monkeypatch.setattr(aqmod, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(aqmod.AqLibraryMissing):
        aqmod.lib()

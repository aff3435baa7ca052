"""The C-ABI library builds, loads without a GPU, exports every function
include/mnw_moe.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "mnw_moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mnw_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import quantized_moe_expert_routed_gb300 as M
    return M.load()


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert len(names) >= 18
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_the_header():
    import quantized_moe_expert_routed_gb300 as M
    assert set(_declared()) == set(M.SIGNATURES)


def test_status_strings(lib):
    assert lib.mnw_status_string(0) == b"ok"
    assert b"workspace" in lib.mnw_status_string(4)


def test_bad_arguments_rejected_before_any_launch(lib):
    # k = 0, E = 0, E too large, T*k too large: rejected on the host
    assert lib.mnw_moe_permute(None, 4, 0, 8, None, None, None, None, 0, None, None, None) == 1
    assert lib.mnw_moe_permute(None, 4, 2, 0, None, None, None, None, 0, None, None, None) == 1
    assert lib.mnw_moe_permute(None, 4, 2, 2000, None, None, None, None, 0, None, None, None) == 1
    assert lib.mnw_moe_permute(None, 1 << 22, 8, 8, None, None, None, None, 0, None, None, None) == 2
    # T = 0 is a no-op
    assert lib.mnw_moe_permute(None, 0, 2, 8, None, None, None, None, 0, None, None, None) == 0
    # quantiser: bad mode, K not a multiple of the group
    assert lib.mnw_moe_quantize_act(0, None, 4, 128, None, 1, None, None, None, None) == 1
    assert lib.mnw_moe_quantize_act(1, None, 4, 100, None, 1, None, None, None, None) == 2
    # combine: H not a multiple of 8
    assert lib.mnw_moe_combine(None, None, None, 2, 2, 12, None, None) == 1
    # GEMM without a layer
    assert lib.mnw_moe_grouped_gemm_w4a16(None, 0, None, None, 4, None, None, None) == 1
    # bounded-wait self-test: null words, limit out of range
    assert lib.mnw_moe_selftest_wait_timeout(1000, None, None, None) == 1
    assert lib.mnw_moe_selftest_wait_timeout(0, ctypes.c_void_p(256), ctypes.c_void_p(512), None) == 1
    # counter-wait self-test: null counter or word, limit out of range
    assert lib.mnw_moe_selftest_counter_timeout(1000, None, 1, ctypes.c_void_p(256), None) == 1
    assert lib.mnw_moe_selftest_counter_timeout(1000, ctypes.c_void_p(256), 1, None, None) == 1
    assert lib.mnw_moe_selftest_counter_timeout(2_000_000, ctypes.c_void_p(256), 1, ctypes.c_void_p(512), None) == 1
    # FP16 row form: K not a multiple of 8, missing factors, R = 0 is a no-op
    assert lib.mnw_moe_quantize_act(3, None, 4, 100, None, 1, None, None, None, None) == 2
    assert lib.mnw_moe_quantize_act(3, ctypes.c_void_p(256), 4, 128, None, 1, ctypes.c_void_p(512), None, None,
                                    None) == 1
    assert lib.mnw_moe_quantize_act(3, None, 0, 128, None, 1, None, None, None, None) == 0
    # FP16-row GEMMs without a layer
    assert lib.mnw_moe_grouped_gemm_w8a16_f16rows(None, 0, None, None, None, 4, None, None, None) == 1
    assert lib.mnw_moe_grouped_gemm_w4a16_f16rows(None, 1, None, None, None, 4, None, None, None) == 1
    # the library's launch counter is readable without a GPU
    assert lib.mnw_moe_launch_count() >= 0


def test_blob_header_checks(lib):
    import synth as S
    hdr = bytearray(S.header_bytes(S.layout(S.FMT_INT4_G128, 4, 256, 256)))
    out = ctypes.c_void_p()
    fake_dev = ctypes.c_void_p(1 << 20)  # 256-aligned, never dereferenced: the header fails first
    bad = bytearray(hdr)
    bad[0] = ord("X")
    assert lib.mnw_moe_layer_init(bytes(bad), fake_dev, 1 << 30, ctypes.byref(out)) == 3
    bad = bytearray(hdr)
    bad[16] ^= 1  # H changed: CRC no longer matches
    assert lib.mnw_moe_layer_init(bytes(bad), fake_dev, 1 << 30, ctypes.byref(out)) == 3
    # misaligned blob pointer
    assert lib.mnw_moe_layer_init(bytes(hdr), ctypes.c_void_p((1 << 20) + 16), 1 << 30, ctypes.byref(out)) == 1


def test_package_fails_loudly_without_its_library(tmp_path):
    """No CPU or PyTorch fallback: with the library absent and no compiler to
    build it, loading the package's library raises."""
    import subprocess
    import sys
    code = f"""
import sys
sys.path.insert(0, {ROOT!r})
import quantized_moe_expert_routed_gb300 as M
from quantized_moe_expert_routed_gb300 import build as B
B.LIB = {str(tmp_path / "libmnw_moe.so")!r}
B.BUILD = {str(tmp_path / "_build")!r}
try:
    M.load()
except RuntimeError as e:
    print("RAISED:", e)
else:
    print("LOADED")
"""
    env = dict(os.environ, NVCC=str(tmp_path / "no-such-nvcc"))
    r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=120)
    assert "RAISED:" in r.stdout and "nvcc not found" in r.stdout, r.stdout + r.stderr


def test_attention_arguments_checked_before_any_launch(lib):
    F = ctypes.c_float
    assert lib.mnw_attn_workspace_size(1, 300, 2, 128) == ((2 * 128 * 304 * 2 + 255) // 256) * 256
    assert lib.mnw_attn_workspace_size(0, 300, 2, 128) == 0
    # B = 0 or T = 0: nothing to do
    assert lib.mnw_attn_prefill(None, None, None, 0, 16, 2, 1, 128, 32, F(0.1), None, None, 0, None, None) == 0
    assert lib.mnw_attn_prefill(None, None, None, 1, 0, 2, 1, 128, 32, F(0.1), None, None, 0, None, None) == 0
    # query heads not a multiple of the kv heads, blk < 1, scale not positive
    assert lib.mnw_attn_prefill(None, None, None, 1, 16, 3, 2, 128, 32, F(0.1), None, None, 0, None, None) == 1
    assert lib.mnw_attn_prefill(None, None, None, 1, 16, 2, 1, 128, 0, F(0.1), None, None, 0, None, None) == 1
    assert lib.mnw_attn_prefill(None, None, None, 1, 16, 2, 1, 128, 32, F(0.0), None, None, 0, None, None) == 1
    assert lib.mnw_attn_prefill(None, None, None, 1, 16, 2, 1, 128, 32, F(float("nan")), None, None, 0, None,
                                None) == 1
    # head dimension other than 128
    assert lib.mnw_attn_prefill(None, None, None, 1, 16, 2, 1, 64, 32, F(0.1), None, None, 0, None, None) == 2
    # null tensors
    assert lib.mnw_attn_prefill(None, None, None, 1, 16, 2, 1, 128, 32, F(0.1), None, None, 0, None, None) == 1

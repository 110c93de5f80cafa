"""CPU-side checks of the C ABI: the library builds, loads and exports every symbol
the header declares; host-only entry points and argument checks work without a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from grok_gqa_attention_gb300 import build
    build.build()
    import grok_gqa_attention_gb300 as G
    return G.load()


def _declared():
    text = open(os.path.join(ROOT, "include", "grok_attn.h")).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(grok_\w+)\s*\(", text, re.M)))


def test_header_declares_the_calls():
    names = _declared()
    for want in ("grok_rope_kv_append", "grok_attn_prefill", "grok_attn_decode", "grok_attn_combine",
                 "grok_attn_decode_workspace", "grok_last_error", "grok_abi_version"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_binding_names_match_header():
    import grok_gqa_attention_gb300 as G
    assert sorted(G.EXPORTS) == _declared()


def test_binding_constants_match_header():
    """The binding's copies of the header's constants (sizes, split, status codes, device bits)."""
    import grok_gqa_attention_gb300 as G
    text = open(os.path.join(ROOT, "include", "grok_attn.h")).read()
    defines = {m.group(1): int(m.group(2), 0) for m in re.finditer(r"^#define (GROK_\w+) (0x[0-9a-fA-F]+|\d+)\b", text, re.M)}
    enums = {m.group(1): int(m.group(2)) for m in re.finditer(r"^\s*(GROK_(?:OK|ERR_\w+)) = (\d+)", text, re.M)}
    pairs = {"N_Q_HEADS": "GROK_N_Q_HEADS", "N_KV_HEADS": "GROK_N_KV_HEADS", "HEAD_DIM": "GROK_HEAD_DIM",
             "DECODE_SPLIT": "GROK_DECODE_SPLIT", "MAX_POSITION": "GROK_MAX_POSITION", "PAGE_TOKENS": "GROK_PAGE_TOKENS",
             "DEV_BAD_START": "GROK_DEV_BAD_START", "DEV_BAD_VALID": "GROK_DEV_BAD_VALID",
             "DEV_BAD_KV_LEN": "GROK_DEV_BAD_KV_LEN", "DEV_TIMEOUT": "GROK_DEV_TIMEOUT", "DEV_BAD_PAGE": "GROK_DEV_BAD_PAGE"}
    for py, c in pairs.items():
        assert getattr(G, py) == defines[c], (py, c)
    for py, c in {"OK": "GROK_OK", "ERR_INVALID_ARG": "GROK_ERR_INVALID_ARG", "ERR_UNSUPPORTED": "GROK_ERR_UNSUPPORTED",
                  "ERR_CUDA": "GROK_ERR_CUDA", "ERR_DEVICE_FAULT": "GROK_ERR_DEVICE_FAULT"}.items():
        assert getattr(G, py) == enums[c], (py, c)


def test_abi_version(lib):
    assert lib.grok_abi_version() == 2


def test_workspace_size_is_host_only(lib):
    n = ctypes.c_size_t(0)
    s = ctypes.c_int(0)
    assert lib.grok_attn_decode_workspace(32, 8192, ctypes.byref(n), ctypes.byref(s)) == 0
    assert s.value == 8192 // 1024          # splits of GROK_DECODE_SPLIT = 1024 keys
    o_bytes = 32 * 8 * 8 * 6 * 128 * 4
    l_bytes = 32 * 8 * 8 * 6 * 4
    assert n.value == o_bytes + ((l_bytes + 255) // 256) * 256
    assert lib.grok_attn_decode_workspace(0, 8192, ctypes.byref(n), ctypes.byref(s)) == 1
    assert lib.grok_attn_decode_workspace(1, 70000, ctypes.byref(n), ctypes.byref(s)) == 1


def test_prefill_minimum_workspace_is_host_only(lib):
    n = ctypes.c_size_t(0)
    assert lib.grok_attn_prefill_workspace_min(1, 8192, ctypes.byref(n)) == 0
    v_half = 8192 * 8 * 128 * 2                      # fp16 copy of V
    flags = (1 + 1 + 9 * 64 * 8 * 3) * 4             # v_flags, list count, fallback list
    assert n.value == ((flags + 255) // 256) * 256 + v_half
    assert lib.grok_attn_prefill_workspace_min(0, 8192, ctypes.byref(n)) == 1
    assert lib.grok_attn_prefill_workspace_min(1, 70000, ctypes.byref(n)) == 1


def test_null_pointers_rejected_before_any_device_call(lib):
    N = None
    assert lib.grok_rope_kv_append(N, N, N, N, 1, 1, 1, N, N, N, N, N) == 1
    assert b"null" in lib.grok_last_error()
    assert lib.grok_attn_prefill(N, N, N, N, N, 1, 1, 1, N, N, N) == 1
    assert lib.grok_attn_decode(N, N, N, N, 1, 1, N, 0, N, N) == 1
    assert lib.grok_attn_combine(N, 0, N, 1, 1, N, N, N) == 1


def test_bad_sizes_rejected(lib):
    p = ctypes.c_void_p(1 << 20)  # never dereferenced: the size check fails first
    assert lib.grok_rope_kv_append(p, p, p, p, 1, 9, 8, p, p, p, None, None) == 1   # T > Tmax
    assert lib.grok_attn_prefill(p, p, p, p, None, 0, 1, 1, p, None, None) == 1     # B = 0


def test_decode_step_workspace_is_host_only(lib):
    n = ctypes.c_size_t(0)
    s = ctypes.c_int(0)
    assert lib.grok_attn_decode_workspace(32, 8192, ctypes.byref(n), ctypes.byref(s)) == 0
    dec = n.value
    assert lib.grok_attn_decode_step_workspace(32, 8192, ctypes.byref(n)) == 0
    q_rot = 32 * 48 * 128 * 2  # the step's q_rot, 256-byte aligned ahead of the split partials
    assert n.value == ((q_rot + 255) // 256) * 256 + dec
    assert lib.grok_attn_decode_step_workspace(0, 8192, ctypes.byref(n)) == 1
    assert lib.grok_attn_decode_step_workspace(1, 70000, ctypes.byref(n)) == 1


def test_new_entry_points_reject_null_pointers_before_any_device_call(lib):
    N = None
    # paged calls, slot insertion and the one-call decode step all check their pointers first
    assert lib.grok_attn_decode_paged(N, N, N, 1, N, 1, N, 1, N, 0, N, N) == 1
    assert lib.grok_attn_prefill_paged(N, N, N, 1, N, 1, N, N, 1, 1, N, N, N) == 1
    assert lib.grok_attn_prefill_ws_paged(N, N, N, 1, N, 1, N, N, 1, 1, N, N, 0, 0, N, N) == 1
    assert lib.grok_rope_kv_append_paged(N, N, N, N, 1, 1, N, N, N, 1, N, 1, N, N) == 1
    assert lib.grok_kv_insert_slot(N, N, 1, 1, 0, N, N, 1, 1, N, 0, N) == 1
    assert lib.grok_attn_decode_step(N, N, N, N, 1, 1, N, N, N, 0, N, N, N) == 1
    assert b"null" in lib.grok_last_error()


def test_misaligned_outputs_rejected_before_any_device_call(lib):
    a32 = ctypes.c_void_p(1 << 20)          # 32-byte aligned, never dereferenced
    a16 = ctypes.c_void_p((1 << 20) + 16)   # 16- but not 32-byte aligned
    assert lib.grok_linear(a32, a32, 256, 64, 256, a16, None, None) == 1
    assert b"32-byte" in lib.grok_last_error()
    assert lib.grok_dequant_int8(a32, a32, 64, 256, a16, None) == 1


def test_linear_tile_widths_rejected_before_any_device_call(lib):
    """N must fill whole 256- or 192-column tiles: 320, 128 and 64 do neither."""
    a32 = ctypes.c_void_p(1 << 20)
    for n in (320, 128, 64, 0):
        assert lib.grok_linear(a32, a32, 256, 64, n, a32, None, None) == 1
        assert b"N of 256 or of 192" in lib.grok_last_error()


def test_product_path_has_no_cpu_route():
    """The binding computes nothing itself: CPU tensors are refused, a missing library
    raises, and no file of the package or its CUDA sources refers to the oracle."""
    import torch

    import grok_gqa_attention_gb300 as G
    q = torch.zeros((1, 4, 48, 128), dtype=torch.bfloat16)
    kv = torch.zeros((1, 4, 8, 128), dtype=torch.bfloat16)
    cache = torch.zeros((1, 8, 8, 128), dtype=torch.bfloat16)
    start = torch.zeros(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        G.rope_kv_append(q, kv, kv, start, torch.empty_like(q), cache, cache.clone())
    with pytest.raises(ValueError, match="CUDA tensor"):
        G.prefill(q, cache, cache, start, None, torch.empty_like(q))
    pkg = os.path.join(ROOT, "grok_gqa_attention_gb300")
    for dirpath, _, files in os.walk(pkg):
        for name in files:
            if name.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, name)).read()
                assert not re.search(r"\boracle\b", text), f"{name} refers to the oracle"


def test_missing_library_raises(monkeypatch, tmp_path):
    import grok_gqa_attention_gb300 as G
    monkeypatch.setattr(G, "_lib", None)
    monkeypatch.setattr(G, "LIB_PATH", str(tmp_path / "libgrok_attn.so"))
    with pytest.raises(RuntimeError, match="missing"):
        G.load()


def test_sticky_cuda_errors_map_to_device_fault(lib):
    """A CUDA error that kills the context is reported as GROK_ERR_DEVICE_FAULT, every
    other failure as GROK_ERR_CUDA (cudaError_t values of the CUDA 13 runtime)."""
    import grok_gqa_attention_gb300 as G
    assert lib.grok_cuda_error_status(0) == G.OK
    sticky = {"illegal address": 700, "launch timeout": 702, "device assert": 710, "hardware stack": 714,
              "illegal instruction": 715, "misaligned address": 716, "invalid address space": 717,
              "invalid pc": 718, "launch failure": 719, "tensor memory leak": 721,
              "uncorrectable ECC": 214, "uncorrectable NVLink": 220, "contained": 226, "external device": 911}
    for what, code in sticky.items():
        assert lib.grok_cuda_error_status(code) == G.ERR_DEVICE_FAULT, what
    recoverable = {"invalid value": 1, "out of memory": 2, "invalid device function": 98,
                   "no device": 100, "not ready": 600, "launch out of resources": 701, "unknown": 999}
    for what, code in recoverable.items():
        assert lib.grok_cuda_error_status(code) == G.ERR_CUDA, what

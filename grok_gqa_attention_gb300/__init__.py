"""Python binding of libgrok_attn.so, the GB300 Grok-1 GQA attention core.

Argument marshalling only: every function takes torch CUDA tensors, checks
their dtype, shape and layout, and passes raw pointers and sizes to the C ABI
declared in include/grok_attn.h. All arithmetic runs in the library's CUDA
kernels; there is no other code path, and every call raises if the library is
not built or the device is not an sm_103 GPU.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

N_Q_HEADS = 48
N_KV_HEADS = 8
HEAD_DIM = 128
DECODE_SPLIT = 1024
MAX_POSITION = 65536

DEV_BAD_START = 0x1
DEV_BAD_VALID = 0x2
DEV_BAD_KV_LEN = 0x4
DEV_TIMEOUT = 0x8
DEV_BAD_PAGE = 0x10

PAGE_TOKENS = 128

# grok_status values (include/grok_attn.h)
OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED = 2
ERR_CUDA = 3
ERR_DEVICE_FAULT = 4

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgrok_attn.so")

EXPORTS = (
    "grok_abi_version",
    "grok_last_error",
    "grok_cuda_error_status",
    "grok_rope_kv_append",
    "grok_rope_kv_append_table",
    "grok_rope_cos_sin",
    "grok_attn_prefill",
    "grok_attn_prefill_workspace",
    "grok_attn_prefill_workspace_min",
    "grok_attn_prefill_ws",
    "grok_attn_decode_workspace",
    "grok_attn_decode",
    "grok_attn_combine",
    "grok_attn_decode_step_static",
    "grok_selftest_bounded_wait",
    "grok_prefill_pipe_create",
    "grok_prefill_pipe_submit",
    "grok_prefill_pipe_wait",
    "grok_prefill_pipe_destroy",
    "grok_qkv_project",
    "grok_qkv_workspace",
    "grok_qkv_rope_append",
    "grok_qkv_rope_append_table",
    "grok_linear",
    "grok_dequant_int8",
    "grok_linear_int8_workspace",
    "grok_linear_int8",
    "grok_rope_kv_append_paged",
    "grok_attn_prefill_paged",
    "grok_attn_prefill_ws_paged",
    "grok_attn_decode_paged",
    "grok_qkv_rope_append_paged",
    "grok_kv_insert_slot",
    "grok_attn_decode_step_workspace",
    "grok_attn_decode_step",
)

_lib: Optional[ctypes.CDLL] = None


class GrokError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"grok status {status}: {message}")
        self.status = status


def load() -> ctypes.CDLL:
    """Load the in-tree library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with grok_gqa_attention_gb300.build.build()")
    lib = ctypes.CDLL(LIB_PATH)
    P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.grok_abi_version.restype = I
    lib.grok_abi_version.argtypes = []
    lib.grok_last_error.restype = ctypes.c_char_p
    lib.grok_last_error.argtypes = []
    lib.grok_cuda_error_status.restype = I
    lib.grok_cuda_error_status.argtypes = [I]
    lib.grok_rope_kv_append.restype = I
    lib.grok_rope_kv_append.argtypes = [P, P, P, P, I, I, I, P, P, P, P, P]
    lib.grok_rope_kv_append_table.restype = I
    lib.grok_rope_kv_append_table.argtypes = [P, P, P, P, I, I, I, P, P, I, P, P, P, P, P]
    lib.grok_rope_cos_sin.restype = I
    lib.grok_rope_cos_sin.argtypes = [I, I, P, P, P]
    lib.grok_attn_prefill.restype = I
    lib.grok_attn_prefill.argtypes = [P, P, P, P, P, I, I, I, P, P, P]
    lib.grok_attn_prefill_workspace.restype = I
    lib.grok_attn_prefill_workspace.argtypes = [I, I, ctypes.POINTER(S)]
    lib.grok_attn_prefill_workspace_min.restype = I
    lib.grok_attn_prefill_workspace_min.argtypes = [I, I, ctypes.POINTER(S)]
    lib.grok_attn_prefill_ws.restype = I
    lib.grok_attn_prefill_ws.argtypes = [P, P, P, P, P, I, I, I, P, P, S, I, P, P]
    lib.grok_attn_decode_workspace.restype = I
    lib.grok_attn_decode_workspace.argtypes = [I, I, ctypes.POINTER(S), ctypes.POINTER(I)]
    lib.grok_attn_decode.restype = I
    lib.grok_attn_decode.argtypes = [P, P, P, P, I, I, P, S, P, P]
    lib.grok_attn_combine.restype = I
    lib.grok_attn_combine.argtypes = [P, S, P, I, I, P, P, P]
    lib.grok_selftest_bounded_wait.restype = I
    lib.grok_selftest_bounded_wait.argtypes = [P, P, ctypes.c_longlong, P]
    lib.grok_attn_decode_step_static.restype = I
    lib.grok_attn_decode_step_static.argtypes = [P, P, P, P, I, I, P, P, P]
    lib.grok_prefill_pipe_create.restype = I
    lib.grok_prefill_pipe_create.argtypes = [I, I, I, P, P, ctypes.POINTER(P)]
    lib.grok_prefill_pipe_submit.restype = I
    lib.grok_prefill_pipe_submit.argtypes = [P, P, P, P, P, P, P]
    lib.grok_prefill_pipe_wait.restype = I
    lib.grok_prefill_pipe_wait.argtypes = [P, ctypes.POINTER(ctypes.c_int32)]
    lib.grok_prefill_pipe_destroy.restype = I
    lib.grok_prefill_pipe_destroy.argtypes = [P]
    lib.grok_qkv_project.restype = I
    lib.grok_qkv_project.argtypes = [P, P, I, P, P, P]
    lib.grok_qkv_workspace.restype = I
    lib.grok_qkv_workspace.argtypes = [I, I, ctypes.POINTER(S)]
    lib.grok_qkv_rope_append.restype = I
    lib.grok_qkv_rope_append.argtypes = [P, P, P, I, I, I, P, P, P, P, S, P, P]
    lib.grok_qkv_rope_append_table.restype = I
    lib.grok_qkv_rope_append_table.argtypes = [P, P, P, I, I, I, P, P, I, P, P, P, P, P]
    lib.grok_linear.restype = I
    lib.grok_linear.argtypes = [P, P, I, I, I, P, P, P]
    lib.grok_dequant_int8.restype = I
    lib.grok_dequant_int8.argtypes = [P, P, I, I, P, P]
    lib.grok_linear_int8_workspace.restype = I
    lib.grok_linear_int8_workspace.argtypes = [I, I, ctypes.POINTER(S)]
    lib.grok_linear_int8.restype = I
    lib.grok_linear_int8.argtypes = [P, P, P, I, I, I, P, P, S, P, P]
    lib.grok_rope_kv_append_paged.restype = I
    lib.grok_rope_kv_append_paged.argtypes = [P, P, P, P, I, I, P, P, P, I, P, I, P, P]
    lib.grok_attn_prefill_paged.restype = I
    lib.grok_attn_prefill_paged.argtypes = [P, P, P, I, P, I, P, P, I, I, P, P, P]
    lib.grok_attn_prefill_ws_paged.restype = I
    lib.grok_attn_prefill_ws_paged.argtypes = [P, P, P, I, P, I, P, P, I, I, P, P, S, I, P, P]
    lib.grok_attn_decode_paged.restype = I
    lib.grok_attn_decode_paged.argtypes = [P, P, P, I, P, I, P, I, P, S, P, P]
    lib.grok_qkv_rope_append_paged.restype = I
    lib.grok_qkv_rope_append_paged.argtypes = [P, P, P, I, I, P, P, P, I, P, I, P, S, P, P]
    lib.grok_kv_insert_slot.restype = I
    lib.grok_kv_insert_slot.argtypes = [P, P, I, I, I, P, P, I, I, P, I, P]
    lib.grok_attn_decode_step_workspace.restype = I
    lib.grok_attn_decode_step_workspace.argtypes = [I, I, ctypes.POINTER(S)]
    lib.grok_attn_decode_step.restype = I
    lib.grok_attn_decode_step.argtypes = [P, P, P, P, I, I, P, P, P, S, P, P, P]
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        msg = load().grok_last_error()
        raise GrokError(status, msg.decode() if msg else "")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _want(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def abi_version() -> int:
    return load().grok_abi_version()


def rope_kv_append(q, k, v, start_pos, q_rot, cache_k, cache_v, dev_status=None, stream=None) -> None:
    """RoPE on q and k; rotated k and raw v written to the caches at start_pos[b] (in place)."""
    B, T = q.shape[0], q.shape[1]
    Tmax = cache_k.shape[1]
    _want(q, "q", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(k, "k", torch.bfloat16, (B, T, N_KV_HEADS, HEAD_DIM))
    _want(v, "v", torch.bfloat16, (B, T, N_KV_HEADS, HEAD_DIM))
    _want(start_pos, "start_pos", torch.int32, (B,))
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_rope_kv_append(_ptr(q), _ptr(k), _ptr(v), _ptr(start_pos), B, T, Tmax, _ptr(q_rot),
                                      _ptr(cache_k), _ptr(cache_v), _ptr(dev_status), _stream(stream)))


def rope_kv_append_table(q, k, v, start_pos, cos_tab, sin_tab, q_rot, cache_k, cache_v, dev_status=None,
                         stream=None) -> None:
    """rope_kv_append with cos/sin read from a table of positions [0, n) (see rope_cos_sin(0, n))."""
    B, T = q.shape[0], q.shape[1]
    Tmax = cache_k.shape[1]
    n = cos_tab.shape[0]
    _want(q, "q", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(k, "k", torch.bfloat16, (B, T, N_KV_HEADS, HEAD_DIM))
    _want(v, "v", torch.bfloat16, (B, T, N_KV_HEADS, HEAD_DIM))
    _want(start_pos, "start_pos", torch.int32, (B,))
    _want(cos_tab, "cos_tab", torch.float32, (n, 64))
    _want(sin_tab, "sin_tab", torch.float32, (n, 64))
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_rope_kv_append_table(_ptr(q), _ptr(k), _ptr(v), _ptr(start_pos), B, T, Tmax, _ptr(cos_tab),
                                            _ptr(sin_tab), n, _ptr(q_rot), _ptr(cache_k), _ptr(cache_v),
                                            _ptr(dev_status), _stream(stream)))


def rope_cos_sin(first_position: int, n_positions: int, stream=None):
    """The fp32 cos/sin table [n_positions, 64] the append kernel uses (new CUDA tensors)."""
    c = torch.empty((n_positions, 64), dtype=torch.float32, device="cuda")
    s = torch.empty_like(c)
    _check(load().grok_rope_cos_sin(int(first_position), int(n_positions), _ptr(c), _ptr(s), _stream(stream)))
    return c, s


def prefill(q_rot, cache_k, cache_v, start_pos, valid_len, out, dev_status=None, stream=None) -> None:
    """Soft-capped causal GQA attention of T new tokens over the cache (valid_len may be None)."""
    B, T = q_rot.shape[0], q_rot.shape[1]
    Tmax = cache_k.shape[1]
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(start_pos, "start_pos", torch.int32, (B,))
    if valid_len is not None:
        _want(valid_len, "valid_len", torch.int32, (B,))
    _want(out, "out", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_attn_prefill(_ptr(q_rot), _ptr(cache_k), _ptr(cache_v), _ptr(start_pos), _ptr(valid_len),
                                    B, T, Tmax, _ptr(out), _ptr(dev_status), _stream(stream)))


def prefill_workspace(B: int, Tmax: int) -> int:
    """Bytes of workspace for prefill_ws() on the current device, with room for the key-range split."""
    n = ctypes.c_size_t(0)
    _check(load().grok_attn_prefill_workspace(B, Tmax, ctypes.byref(n)))
    return n.value


def prefill_workspace_min(B: int, Tmax: int) -> int:
    """Smallest workspace prefill_ws() accepts (fp16 copy of V and flags; calls then run unsplit)."""
    n = ctypes.c_size_t(0)
    _check(load().grok_attn_prefill_workspace_min(B, Tmax, ctypes.byref(n)))
    return n.value


def alloc_prefill_workspace(B: int, Tmax: int, device=None) -> torch.Tensor:
    return torch.empty(prefill_workspace(B, Tmax), dtype=torch.uint8, device=device or "cuda")


def prefill_ws(q_rot, cache_k, cache_v, start_pos, valid_len, out, workspace, dev_status=None, stream=None,
               reuse_v_half: bool = False) -> None:
    """prefill() with fp16 softmax weights and an fp16 copy of V in `workspace` (uint8 CUDA tensor).

    reuse_v_half: rows below start_pos are already in the workspace from earlier calls
    over the same caches (see grok_attn_prefill_ws)."""
    B, T = q_rot.shape[0], q_rot.shape[1]
    Tmax = cache_k.shape[1]
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(start_pos, "start_pos", torch.int32, (B,))
    if valid_len is not None:
        _want(valid_len, "valid_len", torch.int32, (B,))
    _want(out, "out", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(workspace, "workspace", torch.uint8, (workspace.numel(),))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_attn_prefill_ws(_ptr(q_rot), _ptr(cache_k), _ptr(cache_v), _ptr(start_pos),
                                       _ptr(valid_len), B, T, Tmax, _ptr(out), _ptr(workspace), workspace.numel(),
                                       1 if reuse_v_half else 0, _ptr(dev_status), _stream(stream)))


def decode_workspace(B: int, Tmax: int) -> tuple[int, int]:
    """(bytes, splits per sequence) of the workspace decode() needs."""
    n = ctypes.c_size_t(0)
    s = ctypes.c_int(0)
    _check(load().grok_attn_decode_workspace(B, Tmax, ctypes.byref(n), ctypes.byref(s)))
    return n.value, s.value


def alloc_decode_workspace(B: int, Tmax: int, device=None) -> torch.Tensor:
    """A caller-owned workspace tensor for decode()/combine() (256-byte aligned by torch)."""
    nbytes, _ = decode_workspace(B, Tmax)
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def decode(q_rot, cache_k, cache_v, kv_len, workspace, dev_status=None, stream=None) -> None:
    """Split-K part of a decode step: per-split partial sums into the workspace."""
    B, Tmax = cache_k.shape[0], cache_k.shape[1]
    _want(q_rot, "q_rot", torch.bfloat16, (B, N_Q_HEADS, HEAD_DIM))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(kv_len, "kv_len", torch.int32, (B,))
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().grok_attn_decode(_ptr(q_rot), _ptr(cache_k), _ptr(cache_v), _ptr(kv_len), B, Tmax,
                                   _ptr(workspace), nbytes, _ptr(dev_status), _stream(stream)))


def combine(workspace, kv_len, out, Tmax: int, dev_status=None, stream=None) -> None:
    """Combine part of a decode step: out[b, h] = sum of split partials / sum of split row sums."""
    B = out.shape[0]
    _want(kv_len, "kv_len", torch.int32, (B,))
    _want(out, "out", torch.bfloat16, (B, N_Q_HEADS, HEAD_DIM))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().grok_attn_combine(_ptr(workspace), nbytes, _ptr(kv_len), B, Tmax, _ptr(out),
                                    _ptr(dev_status), _stream(stream)))


def selftest_bounded_wait(dev_status, flags, limit_cycles: int, stream=None) -> None:
    """Run the bounded-wait self-test kernel (see grok_selftest_bounded_wait)."""
    _want(dev_status, "dev_status", torch.int32, (1,))
    _want(flags, "flags", torch.int32, (2,))
    _check(load().grok_selftest_bounded_wait(_ptr(dev_status), _ptr(flags), int(limit_cycles), _stream(stream)))


def decode_step_static(q_rot, cache_k, cache_v, kv_len, out, dev_status=None, stream=None) -> None:
    """A decode step that allocates nothing: the library's static workspace holds the partial sums.

    For callers that cannot allocate device memory. Calls that overlap on the
    GPU share that workspace and race; see grok_attn_decode_step_static.
    """
    B, Tmax = cache_k.shape[0], cache_k.shape[1]
    _want(q_rot, "q_rot", torch.bfloat16, (B, N_Q_HEADS, HEAD_DIM))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(kv_len, "kv_len", torch.int32, (B,))
    _want(out, "out", torch.bfloat16, (B, N_Q_HEADS, HEAD_DIM))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_attn_decode_step_static(_ptr(q_rot), _ptr(cache_k), _ptr(cache_v), _ptr(kv_len), B, Tmax,
                                               _ptr(out), _ptr(dev_status), _stream(stream)))


def decode_step(q_rot, cache_k, cache_v, kv_len, workspace, out, dev_status=None, stream=None) -> None:
    """decode() then combine() on the same stream."""
    decode(q_rot, cache_k, cache_v, kv_len, workspace, dev_status, stream)
    combine(workspace, kv_len, out, cache_k.shape[1], dev_status, stream)


def _want_host(t: torch.Tensor, name: str, dtype: torch.dtype, shape: tuple) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def prefill_pipe_create(B: int, T: int, Tmax: int, cache_k, cache_v) -> ctypes.c_void_p:
    """A host-buffer prefill pipeline over the device caches (see grok_prefill_pipe_create)."""
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    h = ctypes.c_void_p()
    _check(load().grok_prefill_pipe_create(int(B), int(T), int(Tmax), _ptr(cache_k), _ptr(cache_v), ctypes.byref(h)))
    return h


def prefill_pipe_submit(pipe, B: int, T: int, q, k, v, start_pos, valid_len, out) -> None:
    """Queue one step from host tensors (page-locked for overlap); out is written by the next wait."""
    _want_host(q, "q", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want_host(k, "k", torch.bfloat16, (B, T, N_KV_HEADS, HEAD_DIM))
    _want_host(v, "v", torch.bfloat16, (B, T, N_KV_HEADS, HEAD_DIM))
    _want_host(start_pos, "start_pos", torch.int32, (B,))
    if valid_len is not None:
        _want_host(valid_len, "valid_len", torch.int32, (B,))
    _want_host(out, "out", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _check(load().grok_prefill_pipe_submit(pipe, _ptr(q), _ptr(k), _ptr(v), _ptr(start_pos), _ptr(valid_len),
                                           _ptr(out)))


def prefill_pipe_wait(pipe) -> int:
    """Block until every queued step finished; returns the OR of their device status bits."""
    st = ctypes.c_int32(0)
    _check(load().grok_prefill_pipe_wait(pipe, ctypes.byref(st)))
    return int(st.value)


def prefill_pipe_destroy(pipe) -> None:
    _check(load().grok_prefill_pipe_destroy(pipe))


MODEL_SIZE = 6144
QKV_COLUMNS = (N_Q_HEADS + 2 * N_KV_HEADS) * HEAD_DIM


def qkv_project(x, w, y, dev_status=None, stream=None) -> None:
    """y [M, 8192] = x [M, 6144] . w [6144, 8192] (bf16, fp32 accumulation)."""
    M = x.shape[0]
    _want(x, "x", torch.bfloat16, (M, MODEL_SIZE))
    _want(w, "w", torch.bfloat16, (MODEL_SIZE, QKV_COLUMNS))
    _want(y, "y", torch.bfloat16, (M, QKV_COLUMNS))
    _check(load().grok_qkv_project(_ptr(x), _ptr(w), M, _ptr(y), _ptr(dev_status), _stream(stream)))


def qkv_workspace(B: int, T: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().grok_qkv_workspace(int(B), int(T), ctypes.byref(n)))
    return int(n.value)


def alloc_qkv_workspace(B: int, T: int, device=None) -> torch.Tensor:
    return torch.empty(qkv_workspace(B, T), dtype=torch.uint8, device=device or "cuda")


def qkv_rope_append(x, w, start_pos, q_rot, cache_k, cache_v, workspace, dev_status=None, stream=None) -> None:
    """Projection fused with RoPE and the cache append (see grok_qkv_rope_append)."""
    B, T = x.shape[0], x.shape[1]
    Tmax = cache_k.shape[1]
    _want(x, "x", torch.bfloat16, (B, T, MODEL_SIZE))
    _want(w, "w", torch.bfloat16, (MODEL_SIZE, QKV_COLUMNS))
    _want(start_pos, "start_pos", torch.int32, (B,))
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_qkv_rope_append(_ptr(x), _ptr(w), _ptr(start_pos), B, T, Tmax, _ptr(q_rot), _ptr(cache_k),
                                       _ptr(cache_v), _ptr(workspace), workspace.numel(), _ptr(dev_status),
                                       _stream(stream)))


def qkv_rope_append_table(x, w, start_pos, cos_tab, sin_tab, q_rot, cache_k, cache_v, dev_status=None,
                          stream=None) -> None:
    """qkv_rope_append with cos/sin from a table of positions [0, n) (see grok_qkv_rope_append_table)."""
    B, T = x.shape[0], x.shape[1]
    Tmax = cache_k.shape[1]
    n = cos_tab.shape[0]
    _want(x, "x", torch.bfloat16, (B, T, MODEL_SIZE))
    _want(w, "w", torch.bfloat16, (MODEL_SIZE, QKV_COLUMNS))
    _want(start_pos, "start_pos", torch.int32, (B,))
    _want(cos_tab, "cos_tab", torch.float32, (n, 64))
    _want(sin_tab, "sin_tab", torch.float32, (n, 64))
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_qkv_rope_append_table(_ptr(x), _ptr(w), _ptr(start_pos), B, T, Tmax, _ptr(cos_tab),
                                             _ptr(sin_tab), n, _ptr(q_rot), _ptr(cache_k), _ptr(cache_v),
                                             _ptr(dev_status), _stream(stream)))


def linear(x, w, y, dev_status=None, stream=None) -> None:
    """y [M, N] = x [M, K] . w [K, N] (bf16 Linear without bias; K % 64 == 0, N % 256 == 0 or N % 192 == 0)."""
    M, K = x.shape
    N = w.shape[1]
    _want(x, "x", torch.bfloat16, (M, K))
    _want(w, "w", torch.bfloat16, (K, N))
    _want(y, "y", torch.bfloat16, (M, N))
    _check(load().grok_linear(_ptr(x), _ptr(w), M, K, N, _ptr(y), _ptr(dev_status), _stream(stream)))


def dequant_int8(w8, scales, w16, stream=None) -> None:
    """w16 [K, N] bf16 = bf16(fp32(w8 [K, N] int8 * scales [N] fp32))."""
    K, N = w8.shape
    _want(w8, "w8", torch.int8, (K, N))
    _want(scales, "scales", torch.float32, (N,))
    _want(w16, "w16", torch.bfloat16, (K, N))
    _check(load().grok_dequant_int8(_ptr(w8), _ptr(scales), K, N, _ptr(w16), _stream(stream)))


def linear_int8_workspace(K: int, N: int) -> int:
    n = ctypes.c_size_t(0)
    _check(load().grok_linear_int8_workspace(int(K), int(N), ctypes.byref(n)))
    return int(n.value)


def linear_int8(x, w8, scales, y, workspace, dev_status=None, stream=None) -> None:
    """y [M, N] = x [M, K] . dequant_int8(w8, scales) (see grok_linear_int8)."""
    M, K = x.shape
    N = w8.shape[1]
    _want(x, "x", torch.bfloat16, (M, K))
    _want(w8, "w8", torch.int8, (K, N))
    _want(scales, "scales", torch.float32, (N,))
    _want(y, "y", torch.bfloat16, (M, N))
    _check(load().grok_linear_int8(_ptr(x), _ptr(w8), _ptr(scales), M, K, N, _ptr(y), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream(stream)))


def _want_pages(k_pool, v_pool, block_table, B: int) -> tuple[int, int]:
    """Checks a paged cache (pools [n_pages, 128, 8, 128], table [B, max_pages]); returns (n_pages, max_pages)."""
    n_pages = k_pool.shape[0]
    _want(k_pool, "k_pool", torch.bfloat16, (n_pages, PAGE_TOKENS, N_KV_HEADS, HEAD_DIM))
    _want(v_pool, "v_pool", torch.bfloat16, (n_pages, PAGE_TOKENS, N_KV_HEADS, HEAD_DIM))
    if block_table.dim() != 2:
        raise ValueError("block_table must be [B, max_pages]")
    max_pages = block_table.shape[1]
    _want(block_table, "block_table", torch.int32, (B, max_pages))
    return n_pages, max_pages


def rope_kv_append_paged(q, k, v, start_pos, q_rot, k_pool, v_pool, block_table, dev_status=None,
                         stream=None) -> None:
    """rope_kv_append into a paged cache: position p of sequence b goes to row p % 128 of page block_table[b, p // 128]."""
    B, T = q.shape[0], q.shape[1]
    _want(q, "q", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(k, "k", torch.bfloat16, (B, T, N_KV_HEADS, HEAD_DIM))
    _want(v, "v", torch.bfloat16, (B, T, N_KV_HEADS, HEAD_DIM))
    _want(start_pos, "start_pos", torch.int32, (B,))
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    n_pages, max_pages = _want_pages(k_pool, v_pool, block_table, B)
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_rope_kv_append_paged(_ptr(q), _ptr(k), _ptr(v), _ptr(start_pos), B, T, _ptr(q_rot),
                                            _ptr(k_pool), _ptr(v_pool), n_pages, _ptr(block_table), max_pages,
                                            _ptr(dev_status), _stream(stream)))


def prefill_paged(q_rot, k_pool, v_pool, block_table, start_pos, valid_len, out, dev_status=None,
                  stream=None) -> None:
    """prefill() over a paged cache (valid_len may be None)."""
    B, T = q_rot.shape[0], q_rot.shape[1]
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    n_pages, max_pages = _want_pages(k_pool, v_pool, block_table, B)
    _want(start_pos, "start_pos", torch.int32, (B,))
    if valid_len is not None:
        _want(valid_len, "valid_len", torch.int32, (B,))
    _want(out, "out", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_attn_prefill_paged(_ptr(q_rot), _ptr(k_pool), _ptr(v_pool), n_pages, _ptr(block_table),
                                          max_pages, _ptr(start_pos), _ptr(valid_len), B, T, _ptr(out),
                                          _ptr(dev_status), _stream(stream)))


def prefill_ws_paged(q_rot, k_pool, v_pool, block_table, start_pos, valid_len, out, workspace, dev_status=None,
                     stream=None, reuse_v_half: bool = False) -> None:
    """prefill_ws() over a paged cache; workspace sized by prefill_workspace(B, block_table.shape[1] * PAGE_TOKENS)."""
    B, T = q_rot.shape[0], q_rot.shape[1]
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    n_pages, max_pages = _want_pages(k_pool, v_pool, block_table, B)
    _want(start_pos, "start_pos", torch.int32, (B,))
    if valid_len is not None:
        _want(valid_len, "valid_len", torch.int32, (B,))
    _want(out, "out", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    _want(workspace, "workspace", torch.uint8, (workspace.numel(),))
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    _check(load().grok_attn_prefill_ws_paged(_ptr(q_rot), _ptr(k_pool), _ptr(v_pool), n_pages, _ptr(block_table),
                                             max_pages, _ptr(start_pos), _ptr(valid_len), B, T, _ptr(out),
                                             _ptr(workspace), workspace.numel(), 1 if reuse_v_half else 0,
                                             _ptr(dev_status), _stream(stream)))


def decode_paged(q_rot, k_pool, v_pool, block_table, kv_len, workspace, dev_status=None, stream=None) -> None:
    """decode() over a paged cache; combine() it with Tmax = block_table.shape[1] * PAGE_TOKENS."""
    B = q_rot.shape[0]
    _want(q_rot, "q_rot", torch.bfloat16, (B, N_Q_HEADS, HEAD_DIM))
    n_pages, max_pages = _want_pages(k_pool, v_pool, block_table, B)
    _want(kv_len, "kv_len", torch.int32, (B,))
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().grok_attn_decode_paged(_ptr(q_rot), _ptr(k_pool), _ptr(v_pool), n_pages, _ptr(block_table),
                                         max_pages, _ptr(kv_len), B, _ptr(workspace), nbytes, _ptr(dev_status),
                                         _stream(stream)))


def qkv_rope_append_paged(x, w, start_pos, q_rot, k_pool, v_pool, block_table, workspace, dev_status=None,
                          stream=None) -> None:
    """qkv_rope_append writing the k and v rows into a paged cache through the block table."""
    B, T = x.shape[0], x.shape[1]
    _want(x, "x", torch.bfloat16, (B, T, MODEL_SIZE))
    _want(w, "w", torch.bfloat16, (MODEL_SIZE, QKV_COLUMNS))
    _want(start_pos, "start_pos", torch.int32, (B,))
    _want(q_rot, "q_rot", torch.bfloat16, (B, T, N_Q_HEADS, HEAD_DIM))
    n_pages, max_pages = _want_pages(k_pool, v_pool, block_table, B)
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().grok_qkv_rope_append_paged(_ptr(x), _ptr(w), _ptr(start_pos), B, T, _ptr(q_rot), _ptr(k_pool),
                                             _ptr(v_pool), n_pages, _ptr(block_table), max_pages, _ptr(workspace),
                                             nbytes, _ptr(dev_status), _stream(stream)))


def kv_insert_slot(cache_k, cache_v, slot: int, src_k, src_v, n_rows: int, step=None, step_value: int = 0,
                   stream=None) -> None:
    """Continuous batching: rows [0, n_rows) of one sequence's caches [L, 8, 128] into batch slot `slot`.

    step (int32 [B], optional) gets step[slot] = step_value.
    """
    B, Tmax = cache_k.shape[0], cache_k.shape[1]
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    L = src_k.shape[0]
    _want(src_k, "src_k", torch.bfloat16, (L, N_KV_HEADS, HEAD_DIM))
    _want(src_v, "src_v", torch.bfloat16, (L, N_KV_HEADS, HEAD_DIM))
    if step is not None:
        _want(step, "step", torch.int32, (B,))
    _check(load().grok_kv_insert_slot(_ptr(cache_k), _ptr(cache_v), B, Tmax, int(slot), _ptr(src_k), _ptr(src_v), L,
                                      int(n_rows), _ptr(step), int(step_value), _stream(stream)))



def decode_step_workspace(B: int, Tmax: int) -> int:
    """Bytes of workspace decode_step_chained() needs (q_rot and the split partials)."""
    n = ctypes.c_size_t(0)
    _check(load().grok_attn_decode_step_workspace(B, Tmax, ctypes.byref(n)))
    return n.value


def alloc_decode_step_workspace(B: int, Tmax: int, device=None) -> torch.Tensor:
    return torch.empty(decode_step_workspace(B, Tmax), dtype=torch.uint8, device=device or "cuda")


def decode_step_chained(q, k, v, start_pos, cache_k, cache_v, workspace, out, dev_status=None, stream=None) -> None:
    """One decode step in one call: append the new token at start_pos, then attend over rows [0, start_pos].

    q [B, 48, 128] (or [B, 1, 48, 128]), k, v [B, 8, 128] (or [B, 1, 8, 128]); the three kernels run as a
    chain of programmatic dependents (see grok_attn_decode_step).
    """
    B, Tmax = cache_k.shape[0], cache_k.shape[1]
    _want(q.view(B, N_Q_HEADS, HEAD_DIM), "q", torch.bfloat16, (B, N_Q_HEADS, HEAD_DIM))
    _want(k.view(B, N_KV_HEADS, HEAD_DIM), "k", torch.bfloat16, (B, N_KV_HEADS, HEAD_DIM))
    _want(v.view(B, N_KV_HEADS, HEAD_DIM), "v", torch.bfloat16, (B, N_KV_HEADS, HEAD_DIM))
    _want(start_pos, "start_pos", torch.int32, (B,))
    _want(cache_k, "cache_k", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(cache_v, "cache_v", torch.bfloat16, (B, Tmax, N_KV_HEADS, HEAD_DIM))
    _want(out, "out", torch.bfloat16, (B, N_Q_HEADS, HEAD_DIM))
    if workspace.device.type != "cuda" or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if dev_status is not None:
        _want(dev_status, "dev_status", torch.int32, (1,))
    nbytes = workspace.numel() * workspace.element_size()
    _check(load().grok_attn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(start_pos), B, Tmax, _ptr(cache_k),
                                        _ptr(cache_v), _ptr(workspace), nbytes, _ptr(out), _ptr(dev_status),
                                        _stream(stream)))

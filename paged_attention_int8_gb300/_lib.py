"""ctypes binding of libpaq8.so: argument marshalling only.

Every step of the computation runs in the library's CUDA kernels; this module
turns torch tensors into pointers, sizes and the current CUDA stream, calls
the C ABI declared in include/paq8.h, and raises on an error status.  There
is no fallback: if the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
import enum
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "_build", "libpaq8.so")
_lock = threading.Lock()
_lib = None


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = 1
    UNSUPPORTED = 2
    CUDA = 3
    DEVICE_CHECK = 4
    TIMEOUT = 5


DEV_BAD_SLOT = 0x1
DEV_BAD_BLOCK = 0x2
DEV_BAD_SEQ = 0x4
DEV_TIMEOUT = 0x8
DEV_BAD_Q = 0x10
DEV_BAD_POS = 0x20

ATTN_NON_CAUSAL = 0x1
ATTN_TEST_TIMEOUT = 0x80000000


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, message: str, bits: int = 0):
        super().__init__(f"{Status(status).name}: {message}")
        self.status = Status(status)
        self.bits = bits


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load libpaq8.so (built by paged_attention_int8_gb300.build)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"libpaq8.so not built ({_LIB_PATH}); run "
                "`python -m paged_attention_int8_gb300.build` (needs nvcc)")
        lib = ctypes.CDLL(_LIB_PATH)
        P, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
        lib.pa_kv_store.argtypes = [P, i64, P, i64, P, i32, i32, i32, P, P, P, P, i32, i32, P, P]
        lib.pa_kv_store.restype = ctypes.c_int
        lib.pa_kv_store_norm_rope.argtypes = [P, i64, P, i64, P, P, i32, i32, i32, P,
                                              ctypes.c_float, P, i32, i32, i32, P, P, P, P, i32,
                                              i32, P, P]
        lib.pa_kv_store_norm_rope.restype = ctypes.c_int
        lib.pa_kv_store_f8v4.argtypes = [P, i64, P, i64, P, i32, i32, i32, P, P, P, P, i32,
                                         i32, P, P]
        lib.pa_kv_store_f8v4.restype = ctypes.c_int
        lib.pa_paged_attention_f8v4.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                                i32, i32, i32, i32, i32, ctypes.c_float, i32, P,
                                                i32, P, P, P, ctypes.c_size_t, ctypes.c_uint32, P]
        lib.pa_paged_attention_f8v4.restype = ctypes.c_int
        lib.pa_auto_num_splits.argtypes = [i32, i32, i32, i32]
        lib.pa_auto_num_splits.restype = i32
        lib.pa_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.pa_workspace_size.restype = ctypes.c_size_t
        lib.pa_paged_attention.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                           i32, i32, i32, i32, ctypes.c_float, i32, P, P, P,
                                           ctypes.c_size_t, ctypes.c_uint32, P]
        lib.pa_paged_attention.restype = ctypes.c_int
        lib.pa_paged_attention_ex.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32,
                                              i32, i32, i32, i32, i32, ctypes.c_float, i32, P,
                                              i32, P, P, P, ctypes.c_size_t, ctypes.c_uint32, P]
        lib.pa_paged_attention_ex.restype = ctypes.c_int
        lib.pa_paged_attention_noalloc.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                   i32, i32, i32, i32, i32, i32,
                                                   ctypes.c_float, i32, P, P, P, P]
        lib.pa_paged_attention_noalloc.restype = ctypes.c_int
        lib.pa_merge_attn_states.argtypes = [P, P, P, P, P, P, i64, i32, P]
        lib.pa_merge_attn_states.restype = ctypes.c_int
        lib.pa_check_status.argtypes = [P, ctypes.POINTER(ctypes.c_uint32), P]
        lib.pa_check_status.restype = ctypes.c_int
        lib.pa_status_string.argtypes = [ctypes.c_int]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_last_error.argtypes = []
        lib.pa_last_error.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _raise_if(status: int):
    if status != Status.OK:
        lib = load()
        msg = lib.pa_last_error().decode() or lib.pa_status_string(status).decode()
        raise PagedAttentionError(status, msg)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device=None):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(*tensors):
    """Every tensor given is a CUDA tensor, and all are on one device (the
    library launches on the current device, so a tensor of another GPU would
    be read through a foreign pointer).  Returns that device."""
    device = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if device is None:
            device = t.device
        elif t.device != device:
            raise ValueError(f"tensors on different devices: {device} and {t.device}")
    return device


def _check16(name, t):
    if t.element_size() != 2:
        raise TypeError(f"{name} must hold 16-bit elements (fp16 scales)")


def _check_cache_shapes(k_cache, k_scale, v_cache, v_scale):
    """K pages token-major, V pages channel-major (see include/paq8.h)."""
    nb, hk, bs, d = k_cache.shape
    want = ((nb, hk, bs, d // 32), (nb, hk, d, bs), (nb, hk, d // 32, bs))
    got = (tuple(k_scale.shape), tuple(v_cache.shape), tuple(v_scale.shape))
    if got != want:
        raise ValueError(f"cache shapes {got} != {want} (k_scale, v_cache, v_scale)")


# ----------------------------------------------------------------------------- API

def kv_store(key, value, slot_mapping, k_cache, k_scale, v_cache, v_scale, status=None,
             stream=None) -> None:
    """Quantize key/value rows [N, Hk, D] (bf16) to q8 and scatter them by
    ``slot_mapping`` (int64 [N]; slot < 0 skipped) into the paged caches:
    ``k_cache`` int8 [num_blocks, Hk, bs, D], ``k_scale`` [num_blocks, Hk, bs, D/32],
    ``v_cache`` int8 [num_blocks, Hk, D, bs], ``v_scale`` [num_blocks, Hk, D/32, bs]
    (scales fp16 or their int16 bits).
    ``status``: optional int32 CUDA tensor (>= 1 element, zeroed) for device checks."""
    device = _check_cuda(key, value, slot_mapping, k_cache, k_scale, v_cache, v_scale, status)
    if key.dtype != torch.bfloat16 or value.dtype != torch.bfloat16:
        raise TypeError("key and value must be bf16")
    if slot_mapping.dtype != torch.int64:
        raise TypeError("slot_mapping must be int64")
    if k_cache.dtype != torch.int8 or v_cache.dtype != torch.int8:
        raise TypeError("caches must be int8")
    _check16("k_scale", k_scale)
    _check16("v_scale", v_scale)
    n, hk, d = key.shape
    if value.shape != key.shape or slot_mapping.shape != (n,):
        raise ValueError("key/value/slot_mapping shapes differ")
    for t in (key, value):
        if t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError("key/value head and channel dims must be contiguous")
    num_blocks, hk2, bs, d2 = k_cache.shape
    if (hk2, d2) != (hk, d):
        raise ValueError("cache shape mismatch")
    _check_cache_shapes(k_cache, k_scale, v_cache, v_scale)
    for t in (k_cache, v_cache, k_scale, v_scale, slot_mapping):
        if not t.is_contiguous():
            raise ValueError("caches and slot_mapping must be contiguous")
    lib = load()
    with torch.cuda.device(device):
        st = lib.pa_kv_store(_ptr(key), key.stride(0), _ptr(value), value.stride(0),
                             _ptr(slot_mapping), n, hk, d, _ptr(k_cache), _ptr(k_scale),
                             _ptr(v_cache), _ptr(v_scale), num_blocks, bs, _ptr(status),
                             _stream(stream, device))
    _raise_if(st)


def kv_store_norm_rope(key, value, slot_mapping, k_cache, k_scale, v_cache, v_scale,
                       positions=None, norm_weight=None, eps: float = 1e-6, rope=None,
                       interleaved: bool = False, status=None, stream=None) -> None:
    """kv_store with each key row normalized and rotated first
    (pa_kv_store_norm_rope): ``norm_weight`` bf16 [D] or None (no norm),
    ``eps`` fp32; ``rope`` fp32 [max_position, rotary_dim / 2, 2] (cos, sin
    per pair) or None (no rotation), ``positions`` int64 [N] the table row of
    each token, ``interleaved`` pairs (2p, 2p + 1) instead of (p, p +
    rotary_dim / 2).  Values are stored as ``kv_store`` stores them."""
    device = _check_cuda(key, value, slot_mapping, k_cache, k_scale, v_cache, v_scale, status,
                         positions, norm_weight, rope)
    if key.dtype != torch.bfloat16 or value.dtype != torch.bfloat16:
        raise TypeError("key and value must be bf16")
    if slot_mapping.dtype != torch.int64 or (positions is not None
                                             and positions.dtype != torch.int64):
        raise TypeError("slot_mapping and positions must be int64")
    n, hk, d = key.shape
    if value.shape != key.shape or slot_mapping.shape != (n,):
        raise ValueError("key/value/slot_mapping shapes differ")
    for t in (key, value):
        if t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError("key/value head and channel dims must be contiguous")
    num_blocks, hk2, bs, d2 = k_cache.shape
    if (hk2, d2) != (hk, d):
        raise ValueError("cache shape mismatch")
    _check_cache_shapes(k_cache, k_scale, v_cache, v_scale)
    if norm_weight is not None and (norm_weight.dtype != torch.bfloat16
                                    or norm_weight.shape != (d,)
                                    or not norm_weight.is_contiguous()):
        raise TypeError("norm_weight must be a contiguous bf16 tensor [head_dim]")
    max_pos, rot = 0, 0
    if rope is not None:
        if rope.dtype != torch.float32 or rope.dim() != 3 or rope.shape[2] != 2 \
                or not rope.is_contiguous():
            raise TypeError("rope must be a contiguous fp32 tensor [max_position, pairs, 2]")
        if positions is None or positions.shape != (n,) or not positions.is_contiguous():
            raise ValueError("a rotation needs int64 positions [num_tokens]")
        max_pos, rot = rope.shape[0], 2 * rope.shape[1]
    lib = load()
    with torch.cuda.device(device):
        st = lib.pa_kv_store_norm_rope(
            _ptr(key), key.stride(0), _ptr(value), value.stride(0), _ptr(slot_mapping),
            _ptr(positions), n, hk, d, _ptr(norm_weight), float(eps), _ptr(rope), max_pos, rot,
            1 if interleaved else 0, _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale),
            num_blocks, bs, _ptr(status), _stream(stream, device))
    _raise_if(st)


def _check_f8v4_shapes(k_cache, v_cache, v_scale, v_zero):
    """fp8 keys [nb, Hk, bs, D] uint8; 4-bit values [nb, Hk, D, bs / 2]
    uint8; scale and zero [nb, Hk, bs] of 16-bit words (see include/paq8.h)."""
    nb, hk, bs, d = k_cache.shape
    want = ((nb, hk, d, bs // 2), (nb, hk, bs), (nb, hk, bs))
    got = (tuple(v_cache.shape), tuple(v_scale.shape), tuple(v_zero.shape))
    if got != want:
        raise ValueError(f"cache shapes {got} != {want} (v_cache, v_scale, v_zero)")
    if k_cache.dtype != torch.uint8 or v_cache.dtype != torch.uint8:
        raise TypeError("fp8 / 4-bit caches: uint8 codes")
    _check16("v_scale", v_scale)
    _check16("v_zero", v_zero)
    for t in (k_cache, v_cache, v_scale, v_zero):
        if not t.is_contiguous():
            raise ValueError("caches must be contiguous")


def kv_store_f8v4(key, value, slot_mapping, k_cache, v_cache, v_scale, v_zero, status=None,
                  stream=None) -> None:
    """Store key/value rows [N, Hk, D] (bf16) in the fp8 / 4-bit format
    (pa_kv_store_f8v4): keys as e4m3, values as 4-bit codes with one fp16
    scale and zero per (token, kv head)."""
    device = _check_cuda(key, value, slot_mapping, k_cache, v_cache, v_scale, v_zero, status)
    if key.dtype != torch.bfloat16 or value.dtype != torch.bfloat16:
        raise TypeError("key and value must be bf16")
    if slot_mapping.dtype != torch.int64 or not slot_mapping.is_contiguous():
        raise TypeError("slot_mapping must be a contiguous int64 tensor")
    n, hk, d = key.shape
    if value.shape != key.shape or slot_mapping.shape != (n,):
        raise ValueError("key/value/slot_mapping shapes differ")
    for t in (key, value):
        if t.stride(2) != 1 or t.stride(1) != d:
            raise ValueError("key/value head and channel dims must be contiguous")
    num_blocks, hk2, bs, d2 = k_cache.shape
    if (hk2, d2) != (hk, d):
        raise ValueError("cache shape mismatch")
    _check_f8v4_shapes(k_cache, v_cache, v_scale, v_zero)
    lib = load()
    with torch.cuda.device(device):
        st = lib.pa_kv_store_f8v4(_ptr(key), key.stride(0), _ptr(value), value.stride(0),
                                  _ptr(slot_mapping), n, hk, d, _ptr(k_cache), _ptr(v_cache),
                                  _ptr(v_scale), _ptr(v_zero), num_blocks, bs, _ptr(status),
                                  _stream(stream, device))
    _raise_if(st)


def paged_attention_f8v4(q, k_cache, v_cache, v_scale, v_zero, cu_seqlens_q, seq_lens,
                         block_table, max_query_len: int, max_seq_len: int,
                         softmax_scale: float | None = None, num_splits: int = 0, out=None,
                         lse=None, workspace=None, stream=None, return_lse: bool = True,
                         causal: bool = True, sinks=None, sliding_window: int = 0,
                         flags: int = 0):
    """paged_attention over the fp8 / 4-bit format (pa_paged_attention_f8v4):
    decode rows only (max_query_len 1).  Other arguments as paged_attention."""
    device = _check_cuda(q, k_cache, v_cache, v_scale, v_zero, cu_seqlens_q, seq_lens,
                         block_table, out, lse, workspace, sinks)
    _check_f8v4_shapes(k_cache, v_cache, v_scale, v_zero)
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise TypeError("q must be a contiguous bf16 tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("seq_lens", seq_lens),
                    ("block_table", block_table)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [S, max_blocks] with unit column stride")
    T, hq, d = q.shape
    num_blocks, hk, bs, d2 = k_cache.shape
    if d2 != d:
        raise ValueError("cache shape mismatch")
    S = seq_lens.shape[0]
    if cu_seqlens_q.shape != (S + 1,) or block_table.shape[0] != S:
        raise ValueError("metadata shapes disagree with seq_lens")
    if sinks is not None and (sinks.dtype != torch.float32 or sinks.shape != (hq,)):
        raise TypeError("sinks must be an fp32 tensor [num_q_heads]")
    if softmax_scale is None:
        softmax_scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    lib = load()
    need = int(lib.pa_workspace_size(S, hq, d, num_splits))
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    flags = int(flags) | (0 if causal else ATTN_NON_CAUSAL)
    with torch.cuda.device(device):
        st = lib.pa_paged_attention_f8v4(
            _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(v_scale), _ptr(v_zero),
            _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(block_table), block_table.stride(0), S, T,
            hq, hk, d, num_blocks, bs, int(max_query_len), int(max_seq_len),
            float(softmax_scale), int(num_splits), _ptr(sinks), int(sliding_window), _ptr(out),
            _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), flags,
            _stream(stream, device))
    _raise_if(st)
    return (out, lse) if return_lse else out


def auto_num_splits(num_seqs: int, num_kv_heads: int, max_query_len: int,
                    max_seq_len: int) -> int:
    return int(load().pa_auto_num_splits(num_seqs, num_kv_heads, max_query_len, max_seq_len))


def workspace_size(num_seqs: int, num_q_heads: int, head_dim: int, num_splits: int = 0) -> int:
    return int(load().pa_workspace_size(num_seqs, num_q_heads, head_dim, num_splits))


def paged_attention(q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens, block_table,
                    max_query_len: int, max_seq_len: int, softmax_scale: float | None = None,
                    num_splits: int = 0, out=None, lse=None, workspace=None, stream=None,
                    return_lse: bool = True, causal: bool = True, sinks=None,
                    sliding_window: int = 0, flags: int = 0):
    """Unified paged attention over the q8 cache (pa_paged_attention_ex).

    q [T, Hq, D] bf16; cu_seqlens_q int32 [S+1]; seq_lens int32 [S] (KV length
    including the new tokens); block_table int32 [S, max_blocks].
    ``max_query_len`` / ``max_seq_len`` are host-side upper bounds (no sync).
    ``causal=False``: every query sees all seq_len keys of its sequence
    (seq_len may be below q_len).  ``sinks``: optional fp32 [Hq] sink logits;
    ``sliding_window``: W > 0 keeps the last W keys of each query (causal
    only).  ``flags``: extra PA_ATTN_* bits (test hooks).
    Returns (out bf16 [T, Hq, D], lse fp32 [T, Hq]) or out alone when
    ``return_lse`` is False.  ``workspace``: optional uint8 CUDA tensor of at
    least ``workspace_size(S, Hq, D, num_splits)`` bytes whose first 4 bytes
    are zero (the device status word); allocated zeroed when omitted."""
    device = _check_cuda(q, workspace, sinks)
    T, hq, d, num_blocks, hk, bs, S, softmax_scale, out, lse = _attention_args(
        q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens, block_table,
        softmax_scale, out, lse, return_lse)
    if sinks is not None and (sinks.dtype != torch.float32 or sinks.shape != (hq,)
                              or not sinks.is_contiguous()):
        raise TypeError("sinks must be a contiguous fp32 tensor [num_q_heads]")
    lib = load()
    need = int(lib.pa_workspace_size(S, hq, d, num_splits))
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=q.device)
    flags = int(flags) | (0 if causal else ATTN_NON_CAUSAL)
    with torch.cuda.device(device):
        st = lib.pa_paged_attention_ex(
            _ptr(q), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale),
            _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(block_table), block_table.stride(0), S, T,
            hq, hk, d, num_blocks, bs, int(max_query_len), int(max_seq_len),
            float(softmax_scale), int(num_splits), _ptr(sinks), int(sliding_window), _ptr(out),
            _ptr(lse), _ptr(workspace), workspace.numel() * workspace.element_size(), flags,
            _stream(stream, device))
    _raise_if(st)
    return (out, lse) if return_lse else out


def paged_attention_noalloc(q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens,
                            block_table, max_query_len: int, max_seq_len: int,
                            softmax_scale: float | None = None, num_splits: int = 0, out=None,
                            lse=None, status=None, stream=None, return_lse: bool = True):
    """paged_attention without a workspace (pa_paged_attention_noalloc): the
    split partials live in the library's fixed 8 MiB device array, so calls
    that overlap on the GPU race, and a split count whose partials do not fit
    is rejected.  ``status``: optional int32 CUDA tensor that receives this
    call's device status bits.  ``out`` / ``lse``, when omitted, are
    allocated here by PyTorch (the library itself allocates nothing)."""
    device = _check_cuda(q, status)
    T, hq, d, num_blocks, hk, bs, S, softmax_scale, out, lse = _attention_args(
        q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens, block_table,
        softmax_scale, out, lse, return_lse)
    if status is not None and (status.dtype != torch.int32 or status.numel() < 1):
        raise TypeError("status must be an int32 tensor")
    with torch.cuda.device(device):
        st = load().pa_paged_attention_noalloc(
            _ptr(q), _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale),
            _ptr(cu_seqlens_q), _ptr(seq_lens), _ptr(block_table), block_table.stride(0), S, T,
            hq, hk, d, num_blocks, bs, int(max_query_len), int(max_seq_len),
            float(softmax_scale), int(num_splits), _ptr(out), _ptr(lse), _ptr(status),
            _stream(stream, device))
    _raise_if(st)
    return (out, lse) if return_lse else out


def _attention_args(q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens,
                    block_table, softmax_scale, out, lse, return_lse):
    """Shared checks of the attention entry points; allocates out / lse when
    omitted."""
    _check_cuda(q, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens, block_table,
                out, lse)
    if q.dtype != torch.bfloat16 or not q.is_contiguous():
        raise TypeError("q must be a contiguous bf16 tensor")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("seq_lens", seq_lens),
                    ("block_table", block_table)):
        if t.dtype != torch.int32:
            raise TypeError(f"{name} must be int32")
    if not (cu_seqlens_q.is_contiguous() and seq_lens.is_contiguous()):
        raise ValueError("cu_seqlens_q and seq_lens must be contiguous")
    if block_table.dim() != 2 or block_table.stride(1) != 1:
        raise ValueError("block_table must be [S, max_blocks] with unit column stride")
    _check16("k_scale", k_scale)
    _check16("v_scale", v_scale)
    T, hq, d = q.shape
    num_blocks, hk, bs, d2 = k_cache.shape
    if d2 != d:
        raise ValueError("cache shape mismatch")
    _check_cache_shapes(k_cache, k_scale, v_cache, v_scale)
    S = seq_lens.shape[0]
    if cu_seqlens_q.shape != (S + 1,) or block_table.shape[0] != S:
        raise ValueError("metadata shapes disagree with seq_lens")
    if softmax_scale is None:
        softmax_scale = d ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((T, hq), dtype=torch.float32, device=q.device)
    return T, hq, d, num_blocks, hk, bs, S, softmax_scale, out, lse


def merge_attn_states(out_a, lse_a, out_b, lse_b, out=None, lse=None, stream=None,
                      return_lse: bool = True):
    """Attention over the union of two disjoint key sets from the attention
    over each: out_a, out_b bf16 [..., D] (e.g. [T, Hq, D]) with their
    natural-log LSEs lse_a, lse_b fp32 [...] (-inf = no key).  ``out`` may be
    out_a or out_b and ``lse`` lse_a or lse_b (in place).  Returns (out, lse)
    or out alone when ``return_lse`` is False."""
    device = _check_cuda(out_a, lse_a, out_b, lse_b, out, lse)
    for name, t in (("out_a", out_a), ("out_b", out_b)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 tensor")
    for name, t in (("lse_a", lse_a), ("lse_b", lse_b)):
        if t.dtype != torch.float32 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous fp32 tensor")
    d = out_a.shape[-1]
    rows = out_a.numel() // d if d else 0
    if out_b.shape != out_a.shape or lse_a.numel() != rows or lse_b.numel() != rows:
        raise ValueError("merge_attn_states: shape mismatch")
    if out is None:
        out = torch.empty_like(out_a)
    elif out.shape != out_a.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise ValueError("out must be a contiguous bf16 tensor shaped like out_a")
    if lse is None and return_lse:
        lse = torch.empty_like(lse_a)
    elif lse is not None and (lse.numel() != rows or lse.dtype != torch.float32
                              or not lse.is_contiguous()):
        raise ValueError("lse must be a contiguous fp32 tensor with one value per row")
    with torch.cuda.device(device):
        st = load().pa_merge_attn_states(_ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b),
                                         _ptr(out), _ptr(lse), rows, d, _stream(stream, device))
    _raise_if(st)
    return (out, lse) if return_lse else out


def check_status(status_tensor, stream=None) -> int:
    """Synchronize, read and clear a device status word (a kv_store status
    tensor or an attention workspace).  Returns the raw bits; raises
    PagedAttentionError when any bit is set."""
    lib = load()
    device = _check_cuda(status_tensor)
    bits = ctypes.c_uint32(0)
    with torch.cuda.device(device):
        st = lib.pa_check_status(_ptr(status_tensor), ctypes.byref(bits),
                                 _stream(stream, device))
    if st == Status.CUDA:
        _raise_if(st)
    if st != Status.OK:
        raise PagedAttentionError(st, lib.pa_status_string(st).decode(), bits.value)
    return bits.value

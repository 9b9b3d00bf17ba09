"""CPU oracle for paged attention over a q8 KV cache.

TEST INFRASTRUCTURE ONLY: only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
never calls it, and it shares no code with the CUDA path.

The arithmetic lives in ``q8_oracle.c`` (plain C: fp32 scalar quantizer, fp64
attention); this module only compiles it with gcc and marshals numpy arrays.
Each function cites the page passage it follows:

* ``q8_quantize_rows`` / ``kv_store`` -- "shared/attention_kit.py"
  (``quantize_q8``) for the format, "shared/kernels/qk_quant_triton.py"
  (``_norm_rope_quant``) for rounding half away from zero, "attention_impl.py"
  (``_store_kvcache_nhd``) for the scatter by slot.
* ``paged_attention`` -- "attention_impl.py" (``_cache_seq``, ``_sdpa_one``,
  ``_prefill_torch_from_cache``) and "triton_turboquant_unified_attention.py"
  (causal limit ``seq_offset <= context_len + query_pos``, GQA row mapping).
* ``attention_partial`` / ``merge_partials`` -- the split-KV segments of
  "triton_turboquant_unified_attention.py" (3D kernel) and the log-sum-exp
  merge ``_merge_lse_`` of "shared/attention_kit.py", in natural-log form.
* ``merge_states`` -- ``_merge_lse_`` of "shared/attention_kit.py" on two
  normalized (out, lse) results, row by row, in natural-log form.
* ``kv_store_f8v4`` and the ``v_zero`` option of ``paged_attention`` -- the
  alternative formats of "triton_turboquant_unified_attention.py" (FP8 keys
  read as e4m3 values; 4-bit values dequantized as idx * scale + zero with
  one fp16 scale and zero per token), stored by a plain quantizer.
* ``norm_rope_rows`` / ``kv_store_norm_rope`` -- the weighted RMSNorm and the
  rotation of "shared/kernels/qk_quant_triton.py" (``_rows``) applied to key
  rows, quantized from fp32 in the q8 format and scattered as ``kv_store``
  does.
* ``paged_attention`` options: attention sinks (USE_SINKS of
  "triton_turboquant_unified_attention.py"), a sliding window
  (``window_size = (sliding_window - 1, 0)`` of "attention_impl.py") and a
  non-causal mode for a cached prefix attended in a pass of its own (the
  two-pass prefix of "shared/attention_kit.py", ``_attend_with_prefix``).

Parity status of each function (what pins it) is listed in the design notes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

# fp-contract=off: no fused multiply-add, so both hosts (x86-64 here, aarch64
# on the GPU machine) round every operation the same way.
CFLAGS = ["-O2", "-std=c11", "-D_GNU_SOURCE", "-ffp-contract=off", "-fno-fast-math",
          "-fPIC", "-shared", "-pthread", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile ``q8_oracle.c`` into ``_build/liboracle.so`` (gcc)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or (
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.or_f32_to_f16_rne.argtypes = [f32]
        lib.or_f32_to_f16_rne.restype = ctypes.c_uint16
        lib.or_f16_to_f32.argtypes = [ctypes.c_uint16]
        lib.or_f16_to_f32.restype = f32
        lib.or_q8_quantize_group.argtypes = [P, P, P]
        lib.or_q8_quantize_group.restype = None
        lib.or_q8_quantize_rows.argtypes = [P, i64, i32, P, P]
        lib.or_q8_quantize_rows.restype = None
        lib.or_kv_store.argtypes = [P, P, P, i64, i32, i32, P, P, P, P, i64, i32, i32]
        lib.or_kv_store.restype = i64
        lib.or_paged_attention.argtypes = [P, i32, i32, i32, i32, P, P, P, P, i64, i32,
                                           P, P, i32, P, i32, f32, P, i64, P, P, i32]
        lib.or_paged_attention.restype = ctypes.c_int
        lib.or_paged_attention_ex.argtypes = [P, i32, i32, i32, i32, P, P, P, P, i64, i32,
                                              P, P, i32, P, i32, f32, P, i32, i32, i32, P, P,
                                              i64, P, P, i32]
        lib.or_paged_attention_ex.restype = ctypes.c_int
        lib.or_attention_partial.argtypes = [P, i32, i32, i32, i32, P, P, P, P, i64, i32,
                                             P, P, i32, P, i32, f32, i32, i32, i64, i64,
                                             P, P, P]
        lib.or_attention_partial.restype = ctypes.c_int
        lib.or_merge_partials.argtypes = [i32, P, P, P, i32, P, P]
        lib.or_merge_partials.restype = None
        lib.or_merge_states.argtypes = [i64, i32, P, P, P, P, P, P]
        lib.or_merge_states.restype = None
        lib.or_f32_to_e4m3.argtypes = [f32]
        lib.or_f32_to_e4m3.restype = ctypes.c_uint8
        lib.or_e4m3_to_f32.argtypes = [ctypes.c_uint8]
        lib.or_e4m3_to_f32.restype = f32
        lib.or_v4_quantize_row.argtypes = [P, i32, P, P, P]
        lib.or_v4_quantize_row.restype = None
        lib.or_kv_store_f8v4.argtypes = [P, P, P, i64, i32, i32, P, P, P, P, i64, i32]
        lib.or_kv_store_f8v4.restype = i64
        lib.or_f32_to_bf16_rne.argtypes = [f32]
        lib.or_f32_to_bf16_rne.restype = ctypes.c_uint16
        lib.or_norm_rope_row.argtypes = [P, i32, P, f32, P, i32, i32, P]
        lib.or_norm_rope_row.restype = None
        lib.or_kv_store_norm_rope.argtypes = [P, P, P, P, i64, i32, i32, P, f32, P, i64, i32,
                                              i32, P, P, P, P, i64, i32, i32]
        lib.or_kv_store_norm_rope.restype = i64
        _lib = lib
        return lib


def _check_cache(kc, ks, vc, vs):
    nb, hk, bs, d = kc.shape
    if d > 1024 or d % 32:
        raise ValueError("head_dim must be a multiple of 32, at most 1024")
    want = ((nb, hk, bs, d // 32), (nb, hk, d, bs), (nb, hk, d // 32, bs))
    if (ks.shape, vc.shape, vs.shape) != want:
        raise ValueError(f"cache shapes {ks.shape, vc.shape, vs.shape} != {want}")


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


# --------------------------------------------------------------------------- formats

def f32_to_f16_bits(x: float) -> int:
    """binary32 -> binary16 bits, round to nearest even (IEEE definition)."""
    return int(_load().or_f32_to_f16_rne(ctypes.c_float(x)))


def f32_to_bf16_bits(x: float) -> int:
    """binary32 -> bfloat16 bits, round to nearest even (IEEE definition)."""
    return int(_load().or_f32_to_bf16_rne(ctypes.c_float(x)))


def f16_bits_to_f32(h: int) -> float:
    return float(_load().or_f16_to_f32(ctypes.c_uint16(h)))


# --------------------------------------------------------------------------- q8

def q8_quantize_group(x: np.ndarray) -> tuple[np.ndarray, int]:
    """One group of 32 fp32 values -> (int8 codes [32], fp16 scale bits)."""
    x = _c(np.asarray(x, dtype=np.float32), np.float32)
    if x.shape != (32,):
        raise ValueError("a q8 group has 32 channels")
    codes = np.empty(32, np.int8)
    scale = np.empty(1, np.uint16)
    _load().or_q8_quantize_group(_ptr(x), _ptr(codes), _ptr(scale))
    return codes, int(scale[0])


def q8_quantize_rows(x_bf16_bits: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """bf16 rows (uint16 bit patterns) [..., D] -> codes int8 [..., D],
    scales fp16 bits uint16 [..., D/32]."""
    x = _c(x_bf16_bits, np.uint16)
    d = x.shape[-1]
    if d % 32:
        raise ValueError("D must be a multiple of 32")
    n = x.size // d
    codes = np.empty(x.shape, np.int8)
    scales = np.empty((*x.shape[:-1], d // 32), np.uint16)
    _load().or_q8_quantize_rows(_ptr(x), n, d, _ptr(codes), _ptr(scales))
    return codes, scales


def kv_store(key_bits, value_bits, slot_mapping, k_cache, k_scale, v_cache, v_scale,
             n_threads: int = 0) -> int:
    """Quantize and scatter [N, Hk, D] bf16 rows into the caches, in place.

    K: codes [num_blocks, Hk, bs, D] int8, scales [num_blocks, Hk, bs, D/32]
    uint16 (fp16 bits).  V pages channel-major: codes [num_blocks, Hk, D, bs],
    scales [num_blocks, Hk, D/32, bs].  Returns the number of skipped
    out-of-range slots."""
    key = _c(key_bits, np.uint16)
    value = _c(value_bits, np.uint16)
    slots = _c(slot_mapping, np.int64)
    for a in (k_cache, v_cache):
        if not (a.flags.c_contiguous and a.dtype == np.int8):
            raise TypeError("code caches must be contiguous int8")
    for a in (k_scale, v_scale):
        if not (a.flags.c_contiguous and a.dtype == np.uint16):
            raise TypeError("scale caches must be contiguous uint16")
    n, hk, d = key.shape
    num_blocks, hk2, bs, d2 = k_cache.shape
    if (hk2, d2) != (hk, d) or value.shape != key.shape or slots.shape != (n,):
        raise ValueError("shape mismatch")
    _check_cache(k_cache, k_scale, v_cache, v_scale)
    return int(_load().or_kv_store(_ptr(key), _ptr(value), _ptr(slots), n, hk, d,
                                   _ptr(k_cache), _ptr(k_scale), _ptr(v_cache),
                                   _ptr(v_scale), num_blocks, bs, n_threads))


# --------------------------------------------------------------------------- fp8 keys, 4-bit values

def f32_to_e4m3_bits(x: float) -> int:
    """binary32 -> fp8 e4m3 bits, round to nearest even, saturating at 448."""
    return int(_load().or_f32_to_e4m3(ctypes.c_float(x)))


def e4m3_bits_to_f32(b: int) -> float:
    return float(_load().or_e4m3_to_f32(ctypes.c_uint8(b)))


def v4_quantize_rows(x_bf16_bits: np.ndarray):
    """Value rows [n, D] (bf16 bits) -> (nibbles uint8 [n, D/2] with channel c
    in byte c/2, low nibble for even c; scale fp16 bits [n]; zero fp16 bits
    [n]): idx = clamp(round_half_away((x - min) / s), 0, 15),
    s = max((max - min) / 15, 1e-8)."""
    x = _c(x_bf16_bits, np.uint16)
    n, d = x.shape
    nib = np.empty((n, d // 2), np.uint8)
    sc = np.empty(n, np.uint16)
    zr = np.empty(n, np.uint16)
    lib = _load()
    for r in range(n):
        lib.or_v4_quantize_row(_ptr(x[r]), d, _ptr(nib[r]), _ptr(sc[r:r + 1]), _ptr(zr[r:r + 1]))
    return nib, sc, zr


def f8v4_cache_shapes(num_blocks: int, hk: int, bs: int, d: int):
    """(k_cache uint8, v_cache uint8, v_scale fp16, v_zero fp16) shapes."""
    return ((num_blocks, hk, bs, d), (num_blocks, hk, d, bs // 2), (num_blocks, hk, bs),
            (num_blocks, hk, bs))


def _check_f8v4(kc, vc, vs, vz):
    nb, hk, bs, d = kc.shape
    want = f8v4_cache_shapes(nb, hk, bs, d)
    if (kc.shape, vc.shape, vs.shape, vz.shape) != want:
        raise ValueError(f"fp8/4-bit cache shapes {kc.shape, vc.shape, vs.shape, vz.shape} != {want}")
    for a, t in ((kc, np.uint8), (vc, np.uint8), (vs, np.uint16), (vz, np.uint16)):
        if not (a.flags.c_contiguous and a.dtype == t):
            raise TypeError("fp8/4-bit caches: contiguous uint8 codes, uint16 scale / zero bits")


def kv_store_f8v4(key_bits, value_bits, slot_mapping, k_cache, v_cache, v_scale, v_zero) -> int:
    """Store [N, Hk, D] bf16 rows in the alternative format: keys as fp8
    e4m3, values as 4-bit codes with one fp16 scale and zero per (token,
    head).  Returns the number of skipped out-of-range slots."""
    key = _c(key_bits, np.uint16)
    value = _c(value_bits, np.uint16)
    slots = _c(slot_mapping, np.int64)
    n, hk, d = key.shape
    _check_f8v4(k_cache, v_cache, v_scale, v_zero)
    num_blocks, hk2, bs, d2 = k_cache.shape
    if (hk2, d2) != (hk, d) or value.shape != key.shape or slots.shape != (n,) or bs % 2:
        raise ValueError("shape mismatch")
    return int(_load().or_kv_store_f8v4(_ptr(key), _ptr(value), _ptr(slots), n, hk, d,
                                        _ptr(k_cache), _ptr(v_cache), _ptr(v_scale),
                                        _ptr(v_zero), num_blocks, bs))


# --------------------------------------------------------------------------- fused store

def _rope_table(rope, rot):
    rope = _c(np.asarray(rope, np.float32), np.float32)
    if rope.ndim != 3 or rope.shape[1:] != (rot // 2, 2):
        raise ValueError("rope must be fp32 [positions, rotary_dim / 2, 2] (cos, sin)")
    return rope


def norm_rope_rows(x_bits, norm_weight_bits=None, eps: float = 1e-6, rope_rows=None,
                   interleaved: bool = False) -> np.ndarray:
    """Key rows [n, D] (bf16 bits) -> the fp32 values the fused store
    quantizes: weighted RMSNorm (norm_weight_bits bf16 bits [D], or None: no
    norm) rounded to bf16, then the rotation of the pairs of rope_rows
    (fp32 [n, rotary_dim / 2, 2]: cos, sin per pair, one row per token; None:
    no rotation), split halves or interleaved pairs ("shared/kernels/
    qk_quant_triton.py", `_rows`)."""
    x = _c(x_bits, np.uint16)
    n, d = x.shape
    if d % 32 or d > 1024:
        raise ValueError("D must be a multiple of 32, at most 1024")
    w = None if norm_weight_bits is None else _c(norm_weight_bits, np.uint16)
    if w is not None and w.shape != (d,):
        raise ValueError("norm weight must hold D values")
    rot = 0
    if rope_rows is not None:
        rope_rows = _c(np.asarray(rope_rows, np.float32), np.float32)
        rot = 2 * rope_rows.shape[1]
        if rope_rows.shape != (n, rot // 2, 2) or rot > d:
            raise ValueError("rope rows must be [n, rotary_dim / 2, 2] with rotary_dim <= D")
    out = np.empty((n, d), np.float32)
    lib = _load()
    for r in range(n):
        lib.or_norm_rope_row(_ptr(x[r]), d, None if w is None else _ptr(w), ctypes.c_float(eps),
                             None if rope_rows is None else _ptr(rope_rows[r]), rot,
                             1 if interleaved else 0, _ptr(out[r]))
    return out


def kv_store_norm_rope(key_bits, value_bits, slot_mapping, positions, k_cache, k_scale,
                       v_cache, v_scale, norm_weight_bits=None, eps: float = 1e-6, rope=None,
                       interleaved: bool = False, n_threads: int = 0) -> int:
    """kv_store with each key row normalized and rotated first (norm_rope_rows
    with the rope row of the token's position; rope fp32 [max_position,
    rotary_dim / 2, 2]) and quantized from the fp32 result; values stored
    unchanged.  Returns the number of skipped rows (slot beyond the cache or
    position outside the table)."""
    key = _c(key_bits, np.uint16)
    value = _c(value_bits, np.uint16)
    slots = _c(slot_mapping, np.int64)
    n, hk, d = key.shape
    num_blocks, hk2, bs, d2 = k_cache.shape
    if (hk2, d2) != (hk, d) or value.shape != key.shape or slots.shape != (n,):
        raise ValueError("shape mismatch")
    _check_cache(k_cache, k_scale, v_cache, v_scale)
    pos = _c(np.zeros(n, np.int64) if positions is None else positions, np.int64)
    w = None if norm_weight_bits is None else _c(norm_weight_bits, np.uint16)
    rot, max_pos, table = 0, 0, None
    if rope is not None:
        table = _c(np.asarray(rope, np.float32), np.float32)
        max_pos, rot = table.shape[0], 2 * table.shape[1]
        table = _rope_table(table, rot)
        if rot > d:
            raise ValueError("rotary_dim must be at most D")
    return int(_load().or_kv_store_norm_rope(
        _ptr(key), _ptr(value), _ptr(slots), _ptr(pos), n, hk, d,
        None if w is None else _ptr(w), ctypes.c_float(eps),
        None if table is None else _ptr(table), max_pos, rot, 1 if interleaved else 0,
        _ptr(k_cache), _ptr(k_scale), _ptr(v_cache), _ptr(v_scale), num_blocks, bs, n_threads))


# --------------------------------------------------------------------------- attention

def _attn_args(q_bits, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens,
               block_table, v_zero=None):
    q = _c(q_bits, np.uint16)
    if v_zero is None:  # q8 caches
        kc, vc = _c(k_cache, np.int8), _c(v_cache, np.int8)
        ks, vs = _c(k_scale, np.uint16), _c(v_scale, np.uint16)
        _check_cache(kc, ks, vc, vs)
    else:               # fp8 keys, 4-bit values (k_scale unused)
        kc, vc = _c(k_cache, np.uint8), _c(v_cache, np.uint8)
        vs, ks = _c(v_scale, np.uint16), _c(v_zero, np.uint16)
        _check_f8v4(kc, vc, vs, ks)
    cu = _c(cu_seqlens_q, np.int32)
    sl = _c(seq_lens, np.int32)
    bt = _c(block_table, np.int32)
    T, hq, d = q.shape
    num_blocks, hk, bs, d2 = kc.shape
    if d2 != d or hq % hk:
        raise ValueError("shape mismatch")
    S = sl.shape[0]
    if cu.shape != (S + 1,) or bt.ndim != 2 or bt.shape[0] != S:
        raise ValueError("metadata shape mismatch")
    keep = (q, kc, ks, vc, vs, cu, sl, bt)
    args = [_ptr(q), T, hq, hk, d, _ptr(kc), _ptr(ks), _ptr(vc), _ptr(vs), num_blocks, bs,
            _ptr(cu), _ptr(sl), S, _ptr(bt), bt.shape[1]]
    return keep, args, T, hq, d


def paged_attention(q_bits, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens,
                    block_table, softmax_scale: float, rows=None, n_threads: int = 0,
                    sinks=None, window: int = 0, causal: bool = True, v_zero=None):
    """fp64 causal paged attention.  Returns (out [n, D] float64, lse [n] float64)
    for the rows ``rows`` (row = token * Hq + q head), all T*Hq rows if None.

    Options (the defaults give plain causal attention): ``sinks`` -- per-q-head
    sink logits [Hq] in the units of the scaled scores, added to the softmax
    denominator only (the USE_SINKS rule of "triton_turboquant_unified_
    attention.py"; the LSE then includes the sink); ``window`` -- sliding
    window W > 0, the query at position p sees keys p - (W - 1) .. p
    ("attention_impl.py", window_size = (sliding_window - 1, 0)), causal
    only; ``causal=False`` -- every query sees all seq_len keys (a cached
    prefix in a pass of its own).  A row with no key and no sink gets out = 0
    and lse = -inf.

    ``v_zero`` (fp16 bits [num_blocks, Hk, bs]) selects the alternative cache
    format of ``kv_store_f8v4``: k_cache holds e4m3 keys, v_cache 4-bit
    values, v_scale / v_zero their per-key scale and zero; k_scale is
    ignored (may be None)."""
    keep, args, T, hq, d = _attn_args(q_bits, k_cache, k_scale, v_cache, v_scale,
                                      cu_seqlens_q, seq_lens, block_table, v_zero)
    if v_zero is not None:
        # the C side reads the zero array from its own argument; k_scale's
        # slot carries nothing for this format
        zero_arr = keep[2]
        args[6] = None
    if rows is None:
        n = T * hq
        rows_arr, rows_ptr = None, None
    else:
        rows_arr = _c(np.asarray(rows, dtype=np.int64), np.int64)
        n = rows_arr.shape[0]
        rows_ptr = _ptr(rows_arr)
    out = np.empty((n, d), np.float64)
    lse = np.empty(n, np.float64)
    if sinks is None and window == 0 and causal and v_zero is None:
        err = _load().or_paged_attention(*args, ctypes.c_float(softmax_scale), rows_ptr, n,
                                         _ptr(out), _ptr(lse), n_threads)
    else:
        sk = None if sinks is None else _c(np.asarray(sinks, np.float32), np.float32)
        if sk is not None and sk.shape != (hq,):
            raise ValueError("sinks must hold one logit per q head")
        err = _load().or_paged_attention_ex(*args, ctypes.c_float(softmax_scale),
                                            None if sk is None else _ptr(sk), int(window),
                                            1 if causal else 0, 0 if v_zero is None else 1,
                                            None if v_zero is None else _ptr(zero_arr),
                                            rows_ptr, n, _ptr(out), _ptr(lse), n_threads)
        del sk
        if err == 2:
            raise ValueError("oracle: window must be >= 0 and needs causal attention")
    del keep
    if err:
        raise RuntimeError("oracle: invalid metadata (block table, seq_lens or cu_seqlens_q)")
    return out, lse


def attention_partial(q_bits, k_cache, k_scale, v_cache, v_scale, cu_seqlens_q, seq_lens,
                      block_table, softmax_scale: float, token: int, head: int, lo: int,
                      hi: int):
    """Partial triple (m, l, acc[D]) of one row over the visible keys in [lo, hi)."""
    keep, args, T, hq, d = _attn_args(q_bits, k_cache, k_scale, v_cache, v_scale,
                                      cu_seqlens_q, seq_lens, block_table)
    m = np.empty(1, np.float64)
    l = np.empty(1, np.float64)
    acc = np.empty(d, np.float64)
    err = _load().or_attention_partial(*args, ctypes.c_float(softmax_scale), token, head,
                                       lo, hi, _ptr(m), _ptr(l), _ptr(acc))
    del keep
    if err:
        raise RuntimeError("oracle: invalid metadata")
    return float(m[0]), float(l[0]), acc


def merge_partials(m, l, acc):
    """Merge partial triples over disjoint key sets -> (out [D], lse)."""
    m = _c(np.asarray(m, np.float64), np.float64)
    l = _c(np.asarray(l, np.float64), np.float64)
    acc = _c(np.asarray(acc, np.float64), np.float64)
    n, d = acc.shape
    out = np.empty(d, np.float64)
    lse = np.empty(1, np.float64)
    _load().or_merge_partials(n, _ptr(m), _ptr(l), _ptr(acc), d, _ptr(out), _ptr(lse))
    return out, float(lse[0])


def merge_states(out_a, lse_a, out_b, lse_b):
    """Row-wise merge of two normalized attention results over disjoint key
    sets: out_a, out_b [rows, D], lse_a, lse_b [rows] (natural log; -inf =
    no key) -> (out [rows, D], lse [rows]), fp64."""
    out_a = _c(np.asarray(out_a, np.float64), np.float64)
    out_b = _c(np.asarray(out_b, np.float64), np.float64)
    lse_a = _c(np.asarray(lse_a, np.float64), np.float64)
    lse_b = _c(np.asarray(lse_b, np.float64), np.float64)
    rows, d = out_a.shape
    if out_b.shape != (rows, d) or lse_a.shape != (rows,) or lse_b.shape != (rows,):
        raise ValueError("merge_states: shape mismatch")
    out = np.empty((rows, d), np.float64)
    lse = np.empty(rows, np.float64)
    _load().or_merge_states(rows, d, _ptr(out_a), _ptr(lse_a), _ptr(out_b), _ptr(lse_b),
                            _ptr(out), _ptr(lse))
    return out, lse

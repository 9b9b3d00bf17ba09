"""Seeded synthetic workloads for paged attention over a q8 KV cache.

This module only draws inputs: sequence lengths, a block table, slot mappings
and bf16 query/key/value rows.  It holds none of the method's arithmetic (no
quantization, no attention) and is the one module that both the oracle tests
and the GPU path use.

Workload shapes follow the pages' serving setting ("attention_impl.py":
`StoreKVCache`, `_forward_mixed_triton` -- prefill chunks first, then decode
tokens; "triton_turboquant_unified_attention.py": `query_start_loc`,
`seq_lens` including the new tokens, `block_table` of int32 page ids).

Draw order for one workload (one ``torch.Generator`` seeded per workload):
lengths, block permutation, per-channel key bias / outlier channels, then K,
V, Q, and finally the padding rows of the store batch.
"""
from __future__ import annotations

import dataclasses
import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Spec:
    """Shape and value recipe of one workload."""
    name: str
    seed: int
    hq: int
    hk: int
    d: int
    bs: int
    # decode sequences: one new token each, KV length uniform in decode_lens
    n_decode: int = 0
    decode_lens: tuple[int, int] = (0, 0)
    # explicit KV lengths of decode sequences (overrides the uniform draw)
    fixed_decode_lens: tuple[int, ...] = ()
    # prefill chunks: prefill_qlen new tokens on a prefix uniform in prefix_lens
    n_prefill: int = 0
    prefill_qlen: int = 0
    prefix_lens: tuple[int, int] = (0, 0)
    # explicit prefix lengths of the prefill chunks (overrides n_prefill and
    # the uniform draw)
    fixed_prefix_lens: tuple[int, ...] = ()
    # key distribution: N(0,1) + per-(kv head, channel) bias of this std,
    # and a fraction of (kv head, channel) slots multiplied by outlier_mult
    k_bias_std: float = 0.0
    k_outlier_frac: float = 0.0
    k_outlier_mult: float = 8.0
    # extra padding rows (slot -1) in the store batch, as a fraction
    pad_frac: float = 0.0
    # split-KV segments the workload asks for: 0 = auto, 1 = none
    num_splits: int = 0
    # spare physical blocks beyond those the sequences use
    spare_blocks: int = 0

    def replace(self, **kw) -> "Spec":
        return dataclasses.replace(self, **kw)


# The five workloads (sizes of the serving scenarios the pages describe).
TINY_DECODE = Spec("tiny_decode", 0, hq=4, hk=2, d=64, bs=16,
                   fixed_decode_lens=(37, 100), num_splits=1)
DECODE_BATCH = Spec("decode_batch", 1, hq=32, hk=8, d=128, bs=16,
                    n_decode=64, decode_lens=(512, 8192), k_bias_std=math.sqrt(2.0))
CHUNKED_PREFILL = Spec("chunked_prefill", 2, hq=32, hk=8, d=128, bs=16,
                       n_prefill=8, prefill_qlen=2048, prefix_lens=(0, 4096),
                       k_outlier_frac=0.01)
MIXED_BATCH = Spec("mixed_batch", 3, hq=64, hk=8, d=128, bs=32,
                   n_prefill=4, prefill_qlen=1024, prefix_lens=(0, 2048),
                   n_decode=128, decode_lens=(1024, 16384), pad_frac=0.02)
LONG_DECODE = Spec("long_decode", 4, hq=32, hk=8, d=128, bs=16,
                   fixed_decode_lens=(131072,) * 8, k_bias_std=math.sqrt(2.0),
                   num_splits=16)
LONG_DECODE_D256 = LONG_DECODE.replace(name="long_decode_d256", seed=5, d=256)

WORKLOADS = {s.name: s for s in (TINY_DECODE, DECODE_BATCH, CHUNKED_PREFILL, MIXED_BATCH,
                                 LONG_DECODE, LONG_DECODE_D256)}


@dataclass
class Workload:
    """Host (CPU) tensors of one workload.

    Sequences are ordered prefill chunks first, then decodes.  All K/V rows of
    a sequence (prefix and new) are drawn; the prefix rows form the
    "populate" store batch and the new rows the per-step store batch.
    """
    spec: Spec
    q_lens: torch.Tensor          # [S] int32
    seq_lens: torch.Tensor        # [S] int32, total KV length incl. new tokens
    cu_seqlens_q: torch.Tensor    # [S+1] int32
    block_table: torch.Tensor     # [S, max_blocks] int32, -1 = unused
    num_blocks: int
    prefix_key: torch.Tensor      # [Np, Hk, D] bf16
    prefix_value: torch.Tensor
    prefix_slots: torch.Tensor    # [Np] int64
    new_key: torch.Tensor         # [Nn, Hk, D] bf16 (new tokens + padding rows)
    new_value: torch.Tensor
    new_slots: torch.Tensor       # [Nn] int64, -1 on padding rows
    q: torch.Tensor               # [T, Hq, D] bf16
    extras: dict = field(default_factory=dict)

    @property
    def num_seqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.q.shape[0])

    @property
    def max_query_len(self) -> int:
        return int(self.q_lens.max().item()) if self.num_seqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max().item()) if self.num_seqs else 0

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.spec.d)

    def all_key_value(self):
        """Every stored row (prefix then new, padding included) as one batch."""
        return (torch.cat([self.prefix_key, self.new_key]),
                torch.cat([self.prefix_value, self.new_value]),
                torch.cat([self.prefix_slots, self.new_slots]))


def _randn_bf16(gen: torch.Generator, shape, chunk_rows: int = 1 << 14) -> torch.Tensor:
    """N(0,1) draws, cast to bf16, produced in row chunks to bound host memory."""
    out = torch.empty(shape, dtype=torch.bfloat16)
    n = shape[0]
    for a in range(0, n, chunk_rows):
        b = min(n, a + chunk_rows)
        out[a:b] = torch.randn((b - a, *shape[1:]), generator=gen, dtype=torch.float32)
    return out


def make_workload(spec: Spec) -> Workload:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(spec.seed)

    # --- lengths: prefill chunks first, then decodes
    q_lens, seq_lens = [], []
    if spec.fixed_prefix_lens:
        for p in spec.fixed_prefix_lens:
            q_lens.append(spec.prefill_qlen)
            seq_lens.append(int(p) + spec.prefill_qlen)
    elif spec.n_prefill:
        lo, hi = spec.prefix_lens
        prefixes = torch.randint(lo, hi + 1, (spec.n_prefill,), generator=gen)
        for p in prefixes.tolist():
            q_lens.append(spec.prefill_qlen)
            seq_lens.append(p + spec.prefill_qlen)
    if spec.fixed_decode_lens:
        for L in spec.fixed_decode_lens:
            q_lens.append(1)
            seq_lens.append(int(L))
    elif spec.n_decode:
        lo, hi = spec.decode_lens
        for L in torch.randint(lo, hi + 1, (spec.n_decode,), generator=gen).tolist():
            q_lens.append(1)
            seq_lens.append(L)
    S = len(seq_lens)
    q_lens_t = torch.tensor(q_lens, dtype=torch.int32)
    seq_lens_t = torch.tensor(seq_lens, dtype=torch.int32)
    cu = torch.zeros(S + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(q_lens_t, 0)

    # --- block table: a random permutation of the physical blocks, dealt in order
    pages = [(L + spec.bs - 1) // spec.bs for L in seq_lens]
    used = sum(pages)
    num_blocks = used + spec.spare_blocks
    perm = torch.randperm(num_blocks, generator=gen)[:used].to(torch.int32)
    max_pages = max(pages) if pages else 1
    block_table = torch.full((S, max_pages), -1, dtype=torch.int32)
    pos = 0
    for s, n in enumerate(pages):
        block_table[s, :n] = perm[pos:pos + n]
        pos += n

    # --- key bias / outlier channels, one draw per (kv head, channel)
    bias = None
    if spec.k_bias_std:
        bias = torch.randn((spec.hk, spec.d), generator=gen) * spec.k_bias_std
    outlier = None
    if spec.k_outlier_frac:
        n_out = max(1, round(spec.k_outlier_frac * spec.hk * spec.d))
        outlier = torch.randperm(spec.hk * spec.d, generator=gen)[:n_out]

    # --- slots of every (sequence, position): page id * bs + offset
    total = sum(seq_lens)
    slots = torch.empty(total, dtype=torch.int64)
    is_new = torch.zeros(total, dtype=torch.bool)
    pos = 0
    for s in range(S):
        L, ql = seq_lens[s], q_lens[s]
        p = torch.arange(L, dtype=torch.int64)
        slots[pos:pos + L] = block_table[s, (p // spec.bs)].to(torch.int64) * spec.bs + p % spec.bs
        is_new[pos + L - ql:pos + L] = True
        pos += L

    # --- K, V, Q
    shape = (total, spec.hk, spec.d)
    key = _randn_bf16(gen, shape)
    if bias is not None or outlier is not None:
        for a in range(0, total, 1 << 14):
            b = min(total, a + (1 << 14))
            part = key[a:b].float()
            if outlier is not None:
                flat = part.view(b - a, spec.hk * spec.d)
                flat[:, outlier] *= spec.k_outlier_mult
            if bias is not None:
                part += bias
            key[a:b] = part.to(torch.bfloat16)
    value = _randn_bf16(gen, shape)
    T = int(cu[-1].item())
    q = _randn_bf16(gen, (T, spec.hq, spec.d))

    new_key, new_value, new_slots = key[is_new], value[is_new], slots[is_new]
    prefix_key, prefix_value, prefix_slots = key[~is_new], value[~is_new], slots[~is_new]
    del key, value

    # --- padding rows (slot -1) at random positions of the store batch
    if spec.pad_frac and new_slots.numel():
        n_pad = max(1, round(spec.pad_frac * new_slots.numel()))
        n_all = new_slots.numel() + n_pad
        pad_pos = torch.randperm(n_all, generator=gen)[:n_pad]
        is_pad = torch.zeros(n_all, dtype=torch.bool)
        is_pad[pad_pos] = True
        pk = _randn_bf16(gen, (n_pad, spec.hk, spec.d))
        pv = _randn_bf16(gen, (n_pad, spec.hk, spec.d))
        k2 = torch.empty((n_all, spec.hk, spec.d), dtype=torch.bfloat16)
        v2 = torch.empty_like(k2)
        s2 = torch.full((n_all,), -1, dtype=torch.int64)
        k2[~is_pad], v2[~is_pad], s2[~is_pad] = new_key, new_value, new_slots
        k2[is_pad], v2[is_pad] = pk, pv
        new_key, new_value, new_slots = k2, v2, s2

    return Workload(spec=spec, q_lens=q_lens_t, seq_lens=seq_lens_t, cu_seqlens_q=cu,
                    block_table=block_table, num_blocks=num_blocks,
                    prefix_key=prefix_key, prefix_value=prefix_value,
                    prefix_slots=prefix_slots, new_key=new_key, new_value=new_value,
                    new_slots=new_slots, q=q)


def cache_shapes(num_blocks: int, hk: int, bs: int, d: int):
    """Shapes of (k_cache, k_scale, v_cache, v_scale).

    K pages are token-major: codes [num_blocks, Hk, bs, D], scales
    [num_blocks, Hk, bs, D/32].  V pages are channel-major: codes
    [num_blocks, Hk, D, bs], scales [num_blocks, Hk, D/32, bs]."""
    return ((num_blocks, hk, bs, d), (num_blocks, hk, bs, d // 32),
            (num_blocks, hk, d, bs), (num_blocks, hk, d // 32, bs))


def empty_cache(num_blocks: int, hk: int, bs: int, d: int, device="cpu", canary: bool = True):
    """Cache tensors (k_cache, k_scale, v_cache, v_scale), shapes as in
    ``cache_shapes``; scales stored as int16 bit patterns of fp16.  With
    ``canary`` the codes are filled with -128 (a value the q8 format never
    produces) and the scales with 0xFFFF (an fp16 NaN), so untouched slots are
    visible."""
    kc, ks, vc, vs = cache_shapes(num_blocks, hk, bs, d)
    fill_c = -128 if canary else 0
    fill_s = -1 if canary else 0
    return (torch.full(kc, fill_c, dtype=torch.int8, device=device),
            torch.full(ks, fill_s, dtype=torch.int16, device=device),
            torch.full(vc, fill_c, dtype=torch.int8, device=device),
            torch.full(vs, fill_s, dtype=torch.int16, device=device))


def cache_shapes_f8v4(num_blocks: int, hk: int, bs: int, d: int):
    """Shapes of (k_cache, v_cache, v_scale, v_zero) in the fp8 / 4-bit
    format: e4m3 keys [num_blocks, Hk, bs, D] (token-major), 4-bit values
    [num_blocks, Hk, D, bs / 2] (channel-major, two keys per byte), fp16
    scale and zero [num_blocks, Hk, bs]."""
    return ((num_blocks, hk, bs, d), (num_blocks, hk, d, bs // 2), (num_blocks, hk, bs),
            (num_blocks, hk, bs))


def empty_cache_f8v4(num_blocks: int, hk: int, bs: int, d: int, device="cpu",
                     canary: bool = True):
    """Cache tensors (k_cache, v_cache, v_scale, v_zero) of the fp8 / 4-bit
    format, shapes as in ``cache_shapes_f8v4``; codes uint8, scale and zero as
    int16 bit patterns of fp16.  With ``canary`` every byte is 0xFF (a NaN
    e4m3 key, which the store never writes for finite inputs below 448)."""
    kc, vc, vs, vz = cache_shapes_f8v4(num_blocks, hk, bs, d)
    fill_c = 0xFF if canary else 0
    fill_s = -1 if canary else 0
    return (torch.full(kc, fill_c, dtype=torch.uint8, device=device),
            torch.full(vc, fill_c, dtype=torch.uint8, device=device),
            torch.full(vs, fill_s, dtype=torch.int16, device=device),
            torch.full(vz, fill_s, dtype=torch.int16, device=device))


def bf16_bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (no arithmetic)."""
    return t.contiguous().view(torch.int16).numpy().view("uint16")


def scale_bits(t: torch.Tensor):
    """int16 scale tensor (fp16 bit patterns) -> numpy uint16."""
    return t.contiguous().cpu().numpy().view("uint16")

"""GPU parity at sizes the oracle finishes in seconds: every output row and
the whole q8 cache compared with the CPU oracle on the same seeded inputs.
Workloads keep the structure of the five serving workloads (decode batches,
chunked prefill on cached prefixes, mixed batches with padding rows, long
split decodes, D = 64/128/256, block sizes 16/32) while spanning several KV
tiles and ragged tails."""
import math

import numpy as np
import pytest
import torch

from paged_attention_int8_gb300 import _lib, inputs
from tests import _harness as H

pytestmark = pytest.mark.gpu

SQRT2 = math.sqrt(2.0)

SMALL = {
    "tiny_decode": inputs.TINY_DECODE,
    "decode": inputs.Spec("small_decode", 101, hq=32, hk=8, d=128, bs=16, n_decode=6,
                          decode_lens=(100, 700), k_bias_std=SQRT2),
    "prefill": inputs.Spec("small_prefill", 102, hq=32, hk=8, d=128, bs=16, n_prefill=3,
                           prefill_qlen=70, prefix_lens=(0, 150), k_outlier_frac=0.01),
    "mixed": inputs.Spec("small_mixed", 103, hq=64, hk=8, d=128, bs=32, n_prefill=2,
                         prefill_qlen=40, prefix_lens=(0, 100), n_decode=5,
                         decode_lens=(50, 400), pad_frac=0.05),
    "long_split": inputs.Spec("small_long", 104, hq=32, hk=8, d=128, bs=16,
                              fixed_decode_lens=(3000, 2500), k_bias_std=SQRT2, num_splits=16),
    "d256": inputs.Spec("small_d256", 105, hq=32, hk=8, d=256, bs=16,
                        fixed_decode_lens=(1500, 900), k_bias_std=SQRT2, num_splits=16),
    "d64_bs32": inputs.Spec("small_d64", 106, hq=4, hk=2, d=64, bs=32, n_prefill=2,
                            prefill_qlen=33, prefix_lens=(0, 70), n_decode=2,
                            decode_lens=(1, 90)),
    "d256_prefill": inputs.Spec("small_d256p", 107, hq=16, hk=4, d=256, bs=32, n_prefill=2,
                                prefill_qlen=45, prefix_lens=(10, 90)),
    "qpk3": inputs.Spec("qpk3", 108, hq=6, hk=2, d=128, bs=16, n_prefill=2, prefill_qlen=50,
                        prefix_lens=(0, 60), n_decode=3, decode_lens=(1, 300)),
    "qpk16": inputs.Spec("qpk16", 109, hq=16, hk=1, d=128, bs=16, n_prefill=1, prefill_qlen=20,
                         prefix_lens=(5, 40), n_decode=3, decode_lens=(20, 200)),
    "qpk1": inputs.Spec("qpk1", 110, hq=8, hk=8, d=64, bs=16, n_prefill=2, prefill_qlen=70,
                        prefix_lens=(0, 30), n_decode=2, decode_lens=(60, 70)),
    "ragged": inputs.Spec("ragged", 111, hq=8, hk=2, d=128, bs=16,
                          fixed_decode_lens=(1, 2, 15, 16, 17, 63, 64, 65, 127, 129)),
}


@pytest.mark.parametrize("name", sorted(SMALL))
def test_small_workload_parity(name, cuda_device):
    w = inputs.make_workload(SMALL[name])
    splits = (None,)
    if w.max_query_len == 1 and w.max_seq_len > 64:
        splits = (None, 1, 2, 16, 0)
    H.check_workload(w, cuda_device, splits=splits)


def test_split_count_does_not_change_results_beyond_rounding(cuda_device):
    w = inputs.make_workload(SMALL["long_split"])
    g = H.GpuState(w, cuda_device)
    outs = {ns: g.attention(num_splits=ns) for ns in (1, 2, 3, 7, 16)}
    base_o, base_l = outs[1]
    for ns, (o, l) in outs.items():
        assert torch.max(torch.abs(o.float() - base_o.float())).item() <= 2e-2
        assert torch.max(torch.abs(l - base_l)).item() <= 1e-4


def _reordered(w: inputs.Workload, order):
    """The same sequences in another order (decodes first, shuffled, ...)."""
    cu = w.cu_seqlens_q.numpy()
    q_parts = [w.q[cu[s]:cu[s + 1]] for s in order]
    q_lens = w.q_lens[order]
    new_cu = torch.zeros(len(order) + 1, dtype=torch.int32)
    new_cu[1:] = torch.cumsum(q_lens, 0)
    return inputs.Workload(spec=w.spec, q_lens=q_lens, seq_lens=w.seq_lens[order],
                           cu_seqlens_q=new_cu, block_table=w.block_table[order].contiguous(),
                           num_blocks=w.num_blocks, prefix_key=w.prefix_key,
                           prefix_value=w.prefix_value, prefix_slots=w.prefix_slots,
                           new_key=w.new_key, new_value=w.new_value, new_slots=w.new_slots,
                           q=torch.cat(q_parts))


def test_mixed_batch_any_order(cuda_device):
    w = inputs.make_workload(SMALL["mixed"])
    S = w.num_seqs
    rng = np.random.default_rng(0)
    for order in (list(range(S))[::-1], list(rng.permutation(S))):
        H.check_workload(_reordered(w, order), cuda_device, splits=(None, 4))


def test_empty_sequences_and_unowned_rows(cuda_device):
    # sequences with no query token (q_len 0), and trailing query rows that no
    # sequence owns: they produce nothing and are left untouched
    w = inputs.make_workload(SMALL["mixed"])
    S = w.num_seqs
    q_lens = torch.cat([w.q_lens[:2], torch.zeros(1, dtype=torch.int32), w.q_lens[2:],
                        torch.zeros(1, dtype=torch.int32)])
    seq_lens = torch.cat([w.seq_lens[:2], torch.tensor([37], dtype=torch.int32), w.seq_lens[2:],
                          torch.tensor([5], dtype=torch.int32)])
    bt = torch.cat([w.block_table[:2], w.block_table[:1], w.block_table[2:], w.block_table[:1]])
    cu = torch.zeros(S + 3, dtype=torch.int32)
    cu[1:] = torch.cumsum(q_lens, 0)
    extra = torch.randn((3, w.spec.hq, w.spec.d)).to(torch.bfloat16)
    w2 = inputs.Workload(spec=w.spec, q_lens=q_lens, seq_lens=seq_lens, cu_seqlens_q=cu,
                         block_table=bt.contiguous(), num_blocks=w.num_blocks,
                         prefix_key=w.prefix_key, prefix_value=w.prefix_value,
                         prefix_slots=w.prefix_slots, new_key=w.new_key, new_value=w.new_value,
                         new_slots=w.new_slots, q=torch.cat([w.q, extra]))
    H.check_workload(w2, cuda_device, splits=(None, 8))


def test_hints_only_steer_tiling(cuda_device):
    # a max_query_len above the real one, and a max_seq_len far above or below
    # the real one, still give the same results
    w = inputs.make_workload(SMALL["mixed"])
    H.check_workload(w, cuda_device, splits=(None,), max_query_len=4 * w.max_query_len)
    H.check_workload(w, cuda_device, splits=(None, 16), max_seq_len=4 * w.max_seq_len)
    H.check_workload(w, cuda_device, splits=(16,), max_seq_len=64)


def test_max_query_len_below_a_q_len_is_flagged(cuda_device):
    # the decode-only path cannot serve a multi-token sequence: it says so
    w = inputs.make_workload(SMALL["mixed"])
    g = H.GpuState(w, cuda_device)
    ws = torch.zeros(_lib.workspace_size(w.num_seqs, w.spec.hq, w.spec.d, 0), dtype=torch.uint8,
                     device=cuda_device)
    _lib.paged_attention(g.q, g.kc, g.ks, g.vc, g.vs, g.cu, g.seq_lens, g.block_table, 1,
                         w.max_seq_len, workspace=ws)
    with pytest.raises(_lib.PagedAttentionError) as e:
        _lib.check_status(ws)
    assert e.value.bits == _lib.DEV_BAD_SEQ


def test_no_lse_requested(cuda_device):
    w = inputs.make_workload(SMALL["decode"])
    g = H.GpuState(w, cuda_device)
    o = H.OracleState(w)
    rows = H.owned_rows(w)
    ref_out, ref_lse = o.attention(rows=rows)
    out, _ = g.attention(lse=False)
    H.compare(out, None, ref_out, ref_lse, rows)


def test_one_key_rows(cuda_device):
    # first token of a prefill with no prefix, and single-key decodes: the
    # output is the dequantized value row and the LSE its score
    spec = inputs.Spec("one_key", 112, hq=8, hk=2, d=128, bs=16, n_prefill=2, prefill_qlen=17,
                       prefix_lens=(0, 0), fixed_decode_lens=(1, 1))
    H.check_workload(inputs.make_workload(spec), cuda_device, splits=(None, 16))


# ------------------------------------------------------------------ kv_store alone

def test_kv_store_bit_exact_with_padding_and_strided_rows(cuda_device):
    w = inputs.make_workload(SMALL["mixed"])
    g = H.GpuState(w, cuda_device, populate=False)
    # rows as a slice of a wider [N, 3, Hk, D] tensor (e.g. a fused qkv buffer)
    k, v, slots = w.all_key_value()
    wide = torch.zeros((k.shape[0], 3, w.spec.hk, w.spec.d), dtype=torch.bfloat16)
    wide[:, 1] = k
    wide[:, 2] = v
    wide = wide.to(cuda_device)
    _lib.kv_store(wide[:, 1], wide[:, 2], slots.to(cuda_device), g.kc, g.ks, g.vc, g.vs,
                  status=g.status)
    assert _lib.check_status(g.status) == 0
    H.assert_cache_equal(g, H.OracleState(w))


def test_kv_store_adversarial_values(cuda_device):
    # ties on the scale-one grid, one huge outlier over tiny values, all-zero
    # groups, subnormal-range scales: codes and scales bit-exact
    rng = np.random.default_rng(3)
    n, hk, d, bs = 64, 2, 128, 16
    x = rng.standard_normal((n, hk, d))
    x[0::4] = rng.integers(-126, 127, size=x[0::4].shape) + 0.5
    x[0::4, :, ::32] = 127.0
    x[1::4] *= 1e-3
    x[1::4, :, 5] = 900.0
    x[2::4, :, 32:64] = 0.0
    x[3::4] *= 1e-6
    key = torch.from_numpy(x).to(torch.bfloat16)
    value = torch.from_numpy(-x[::-1].copy()).to(torch.bfloat16)
    slots = torch.from_numpy(rng.permutation(n * 2)[:n].astype(np.int64))
    spec = inputs.Spec("adv", 0, hq=hk, hk=hk, d=d, bs=bs)
    empty = inputs.Workload(spec=spec, q_lens=torch.zeros(0, dtype=torch.int32),
                            seq_lens=torch.zeros(0, dtype=torch.int32),
                            cu_seqlens_q=torch.zeros(1, dtype=torch.int32),
                            block_table=torch.zeros((0, 1), dtype=torch.int32), num_blocks=8,
                            prefix_key=key, prefix_value=value, prefix_slots=slots,
                            new_key=key[:0], new_value=value[:0], new_slots=slots[:0],
                            q=torch.zeros((0, hk, d), dtype=torch.bfloat16))
    g = H.GpuState(empty, cuda_device)
    H.assert_cache_equal(g, H.OracleState(empty))


def _store_only_workload(key, value, slots, num_blocks, bs):
    hk, d = key.shape[1], key.shape[2]
    spec = inputs.Spec("store_only", 0, hq=hk, hk=hk, d=d, bs=bs)
    return inputs.Workload(spec=spec, q_lens=torch.zeros(0, dtype=torch.int32),
                           seq_lens=torch.zeros(0, dtype=torch.int32),
                           cu_seqlens_q=torch.zeros(1, dtype=torch.int32),
                           block_table=torch.zeros((0, 1), dtype=torch.int32),
                           num_blocks=num_blocks, prefix_key=key, prefix_value=value,
                           prefix_slots=slots, new_key=key[:0], new_value=value[:0],
                           new_slots=slots[:0], q=torch.zeros((0, hk, d), dtype=torch.bfloat16))


def test_kv_store_near_ties_bit_exact(cuda_device):
    # values whose quotient x / s lies at or within a few fp32 ulps of a
    # rounding tie k + 1/2, for scales that are not powers of two: the codes
    # must still equal those of the IEEE quotient (the oracle's rule)
    rng = np.random.default_rng(11)
    n, hk, d, bs = 512, 2, 128, 16
    amax = rng.uniform(0.05, 80.0, size=(n, hk, d // 32)).astype(np.float32)
    amax = torch.from_numpy(amax).to(torch.bfloat16).float().numpy()  # representable
    s = np.maximum(amax / np.float32(127.0), np.float32(1e-8)).astype(np.float32)
    k = rng.integers(-126, 126, size=(n, hk, d)).astype(np.float64)
    eps = rng.choice([0.0, 2.0 ** -20, -(2.0 ** -20), 2.0 ** -13, -(2.0 ** -13), 2.0 ** -9],
                     size=(n, hk, d))
    x = (k + 0.5 + eps) * np.repeat(s, 32, axis=2).astype(np.float64)
    x[:, :, ::32] = amax  # the group max
    key = torch.from_numpy(x).to(torch.bfloat16)
    value = torch.from_numpy(-x).to(torch.bfloat16)
    slots = torch.from_numpy(rng.permutation(n)[:n].astype(np.int64))
    w = _store_only_workload(key, value, slots, n // bs, bs)
    g = H.GpuState(w, cuda_device)
    H.assert_cache_equal(g, H.OracleState(w))


def _page_run_batches(rng, hk, d, bs, nb):
    """Two store batches over sequences laid on randomly permuted blocks,
    each sequence starting mid-page (as a prefill chunk after a prefix or a
    cache population) and cut in two, so that the second batch continues
    pages the first left partial; about 8% padding rows and a few scattered
    single slots are mixed into both."""
    perm = list(rng.permutation(nb))
    a_slots, b_slots = [], []
    for L in rng.integers(3, 5 * bs, size=10):
        start = int(rng.integers(0, bs))
        nblk = (start + int(L) + bs - 1) // bs
        blocks = [perm.pop() for _ in range(nblk)]
        seq = [blocks[p // bs] * bs + p % bs for p in range(start, start + int(L))]
        cut = int(rng.integers(0, len(seq) + 1))
        a_slots += seq[:cut]
        b_slots += seq[cut:]
    spare = [perm.pop() * bs + int(rng.integers(0, bs)) for _ in range(6)]
    a_slots += spare[:3]
    b_slots += spare[3:]
    out = []
    for sl in (a_slots, b_slots):
        sl = np.array(sl, np.int64)
        at = rng.integers(0, sl.shape[0] + 1, size=max(1, sl.shape[0] // 12))
        full = np.insert(sl, np.sort(at), -1)
        n = full.shape[0]
        k = torch.from_numpy(rng.standard_normal((n, hk, d)) * 1.5).to(torch.bfloat16)
        v = torch.from_numpy(rng.standard_normal((n, hk, d))).to(torch.bfloat16)
        out.append((k, v, torch.from_numpy(full)))
    return out


@pytest.mark.parametrize("d,bs", [(64, 16), (128, 16), (128, 32), (256, 16), (256, 32)])
def test_kv_store_page_runs_bit_exact(d, bs, cuda_device):
    rng = np.random.default_rng(50 + d + bs)
    hk, nb = 2, 128
    (ka, va, sa), (kb, vb, sb) = _page_run_batches(rng, hk, d, bs, nb)
    spec = inputs.Spec("page_runs", 0, hq=hk, hk=hk, d=d, bs=bs)
    w = inputs.Workload(spec=spec, q_lens=torch.zeros(0, dtype=torch.int32),
                        seq_lens=torch.zeros(0, dtype=torch.int32),
                        cu_seqlens_q=torch.zeros(1, dtype=torch.int32),
                        block_table=torch.zeros((0, 1), dtype=torch.int32), num_blocks=nb,
                        prefix_key=ka, prefix_value=va, prefix_slots=sa,
                        new_key=kb, new_value=vb, new_slots=sb,
                        q=torch.zeros((0, hk, d), dtype=torch.bfloat16))
    g = H.GpuState(w, cuda_device)  # stores batch a, then batch b
    H.assert_cache_equal(g, H.OracleState(w))


def _near_tie_groups(rng, count):
    """Groups of 32 bf16 values (as fp32), group max first, whose quotients
    x / s (s = fp32(amax / 127)) sit on a rounding tie k + 1/2 or close to
    one: half the groups have a power-of-two scale (amax = 1.984375 * 2^e,
    so s = 2^(e-6)) and exact ties x = (k + 1/2) s; the rest have other
    scales and values searched among all bf16 numbers for |x / s - (k +
    1/2)| < 2^-12 (fp32 quotient)."""
    pos = (np.arange(0x0080, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    groups = []
    while len(groups) < count:
        if len(groups) % 2 == 0:
            e = int(rng.integers(-6, 7))
            amax = np.float32(1.984375 * 2.0 ** e)
            s = np.float32(amax / np.float32(127.0))
            k = rng.integers(-127, 127, size=31)
            vals = ((k + 0.5) * np.float64(s)).astype(np.float32)
        else:
            amax = np.float32(torch.tensor(float(rng.uniform(0.05, 60.0))).to(torch.bfloat16).item())
            s = np.float32(amax / np.float32(127.0))
            cand = pos[pos < amax]
            q = (cand / s).astype(np.float32)
            near = np.abs(q - np.floor(q) - 0.5) < 2.0 ** -12
            if near.sum() < 4:
                continue
            pick = rng.choice(cand[near], size=31)
            vals = pick * rng.choice([-1.0, 1.0], size=31).astype(np.float32)
        groups.append(np.concatenate([[amax], vals]).astype(np.float32))
    return np.stack(groups)


def test_kv_store_exact_and_near_ties_bit_exact(cuda_device):
    rng = np.random.default_rng(12)
    n, hk, d, bs = 128, 2, 128, 16
    G = d // 32
    gk = _near_tie_groups(rng, n * hk * G)
    gv = _near_tie_groups(rng, n * hk * G)
    key = torch.from_numpy(gk.reshape(n, hk, d)).to(torch.bfloat16)
    value = torch.from_numpy(gv.reshape(n, hk, d)).to(torch.bfloat16)
    assert torch.equal(key.float(), torch.from_numpy(gk.reshape(n, hk, d)))  # exact in bf16
    slots = torch.from_numpy(rng.permutation(n).astype(np.int64))
    w = _store_only_workload(key, value, slots, n // bs, bs)
    g = H.GpuState(w, cuda_device)
    H.assert_cache_equal(g, H.OracleState(w))


# ------------------------------------------------------------------ device checks

def test_kv_store_flags_out_of_range_slot(cuda_device):
    H.ensure_built()
    kc, ks, vc, vs = inputs.empty_cache(2, 1, 16, 64, device=cuda_device)
    st = torch.zeros(4, dtype=torch.int32, device=cuda_device)
    key = torch.ones((3, 1, 64), dtype=torch.bfloat16, device=cuda_device)
    slots = torch.tensor([3, 32, -1], dtype=torch.int64, device=cuda_device)
    _lib.kv_store(key, key, slots, kc, ks, vc, vs, status=st)
    with pytest.raises(_lib.PagedAttentionError) as e:
        _lib.check_status(st)
    assert e.value.bits == _lib.DEV_BAD_SLOT
    codes = kc.cpu().reshape(32, 64)
    assert torch.all(codes[3] == 127)
    assert torch.all(codes[torch.arange(32) != 3] == -128)
    assert _lib.check_status(st) == 0  # read-and-clear


def test_attention_flags_bad_block_table_and_bad_lengths(cuda_device):
    w = inputs.make_workload(SMALL["decode"])
    g = H.GpuState(w, cuda_device)
    bt = g.block_table.clone()
    bt[1, 3] = w.num_blocks + 7
    bt[2, 0] = -5
    ws = torch.zeros(_lib.workspace_size(w.num_seqs, w.spec.hq, w.spec.d, 4), dtype=torch.uint8,
                     device=cuda_device)
    _lib.paged_attention(g.q, g.kc, g.ks, g.vc, g.vs, g.cu, g.seq_lens, bt, 1, w.max_seq_len,
                         num_splits=4, workspace=ws)
    with pytest.raises(_lib.PagedAttentionError) as e:
        _lib.check_status(ws)
    assert e.value.bits & _lib.DEV_BAD_BLOCK
    # seq_len < q_len
    sl = g.seq_lens.clone()
    cu = torch.tensor([0, 3, 4], dtype=torch.int32, device=cuda_device)
    sl2 = torch.tensor([2, int(sl[1])], dtype=torch.int32, device=cuda_device)
    _lib.paged_attention(g.q[:4], g.kc, g.ks, g.vc, g.vs, cu, sl2, g.block_table[:2], 3,
                         w.max_seq_len, workspace=ws)
    with pytest.raises(_lib.PagedAttentionError) as e:
        _lib.check_status(ws)
    assert e.value.bits & _lib.DEV_BAD_SEQ
    # the context is still usable: a clean run afterwards passes
    o = H.OracleState(w)
    rows = H.owned_rows(w)
    ref_out, ref_lse = o.attention(rows=rows)
    out, lse = g.attention()
    H.compare(out, lse, ref_out, ref_lse, rows)


def test_workspace_reused_across_calls(cuda_device):
    # one workspace for calls of different shapes and split counts: nothing a
    # call leaves in it (split partials, a cleared status word) changes the next
    ws = torch.zeros(_lib.workspace_size(16, 32, 128, 16), dtype=torch.uint8, device=cuda_device)
    for name, ns in (("decode", 16), ("long_split", 4), ("decode", 2), ("long_split", 16)):
        w = inputs.make_workload(SMALL[name])
        g = H.GpuState(w, cuda_device)
        o = H.OracleState(w)
        rows = H.owned_rows(w)
        ref_out, ref_lse = o.attention(rows=rows)
        for _ in range(2):
            out = torch.full_like(g.q, float("nan"))
            lse = torch.full((w.num_tokens, w.spec.hq), float("nan"), device=cuda_device)
            _lib.paged_attention(g.q, g.kc, g.ks, g.vc, g.vs, g.cu, g.seq_lens, g.block_table,
                                 w.max_query_len, w.max_seq_len, w.softmax_scale,
                                 num_splits=ns, out=out, lse=lse, workspace=ws)
            assert _lib.check_status(ws) == 0
            H.compare(out, lse, ref_out, ref_lse, rows, label=f"{name} splits={ns} reused")

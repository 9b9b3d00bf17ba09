"""The seeded input generators against the recipe they claim: block tables
that are permutations of the physical blocks, slots that follow the block
table, the per-channel key bias of variance 2, exactly round(1 % of Hk * D)
outlier channels scaled by 8, the padding-row fraction, length ranges and
determinism.  Small variants of the serving workloads keep this on the CPU
in seconds."""
import math

import numpy as np
import pytest
import torch

from paged_attention_int8_gb300 import inputs

VARIANTS = [
    inputs.TINY_DECODE,
    inputs.DECODE_BATCH.replace(name="decode_small", n_decode=6, decode_lens=(512, 900)),
    inputs.CHUNKED_PREFILL.replace(name="prefill_small", n_prefill=3, prefill_qlen=64,
                                   prefix_lens=(0, 300)),
    inputs.MIXED_BATCH.replace(name="mixed_small", n_prefill=2, prefill_qlen=64,
                               prefix_lens=(0, 100), n_decode=6, decode_lens=(40, 300)),
]


@pytest.mark.parametrize("spec", VARIANTS, ids=lambda s: s.name)
def test_block_table_slots_and_lengths(spec):
    w = inputs.make_workload(spec)
    bt = w.block_table.numpy()
    lens = w.seq_lens.numpy()
    qls = w.q_lens.numpy()
    pages = -(-lens // spec.bs)
    used = np.concatenate([bt[s, :n] for s, n in enumerate(pages)])
    assert used.size == pages.sum() == len(set(used.tolist()))          # each block once
    assert used.min() >= 0 and used.max() < w.num_blocks
    for s, n in enumerate(pages):
        assert np.all(bt[s, n:] == -1)                                   # unused entries
    # q lengths and KV lengths per the spec (prefill chunks first, then decodes)
    n_pre = spec.n_prefill
    assert np.all(qls[:n_pre] == spec.prefill_qlen) and np.all(qls[n_pre:] == 1)
    if spec.fixed_decode_lens:
        assert tuple(lens[n_pre:]) == spec.fixed_decode_lens
    elif spec.n_decode:
        lo, hi = spec.decode_lens
        assert np.all((lens[n_pre:] >= lo) & (lens[n_pre:] <= hi))
    if n_pre:
        lo, hi = spec.prefix_lens
        pre = lens[:n_pre] - qls[:n_pre]
        assert np.all((pre >= lo) & (pre <= hi))
    assert np.array_equal(w.cu_seqlens_q.numpy(), np.concatenate([[0], np.cumsum(qls)]))
    # slots follow the block table: token j of sequence s -> bt[s, j // bs] * bs + j % bs;
    # the prefix batch holds positions < L - q_len, the new batch the rest
    pre_slots, new_slots = [], []
    for s in range(w.num_seqs):
        j = np.arange(lens[s])
        sl = bt[s, j // spec.bs].astype(np.int64) * spec.bs + j % spec.bs
        pre_slots.append(sl[:lens[s] - qls[s]])
        new_slots.append(sl[lens[s] - qls[s]:])
    assert np.array_equal(w.prefix_slots.numpy(), np.concatenate(pre_slots))
    got_new = w.new_slots.numpy()
    assert np.array_equal(got_new[got_new >= 0], np.concatenate(new_slots))
    n_pad = int(np.sum(got_new < 0))
    n_real = int(np.sum(got_new >= 0))
    assert n_pad == (max(1, round(spec.pad_frac * n_real)) if spec.pad_frac else 0)
    assert w.q.shape == (int(qls.sum()), spec.hq, spec.d)
    assert w.new_key.shape[0] == got_new.shape[0] == w.new_value.shape[0]


def test_generation_is_deterministic_per_seed():
    spec = VARIANTS[3]
    a, b = inputs.make_workload(spec), inputs.make_workload(spec)
    for name in ("q", "prefix_key", "prefix_value", "new_key", "new_value", "new_slots",
                 "block_table", "seq_lens"):
        assert torch.equal(getattr(a, name), getattr(b, name)), name
    c = inputs.make_workload(spec.replace(seed=spec.seed + 1))
    assert not torch.equal(a.q, c.q)


def _all_keys(w):
    return torch.cat([w.prefix_key, w.new_key[w.new_slots >= 0]]).float()


def test_key_bias_has_variance_two_per_head_and_channel():
    # "k ~ N(0,1) plus a per-channel bias ~N(0,2)": one bias per (kv head,
    # channel), shared by all tokens, variance 2
    spec = inputs.DECODE_BATCH.replace(name="bias_check", n_decode=3, decode_lens=(1500, 1600))
    w = inputs.make_workload(spec)
    k = _all_keys(w)                                   # [N, hk, d]
    mean = k.mean(dim=0)                               # ~ the bias, +- 1/sqrt(N)
    resid = (k - mean).std(dim=0)                      # ~ 1 everywhere
    n_slots = spec.hk * spec.d
    var = float(mean.var())
    assert abs(var - 2.0) < 4 * 2.0 * math.sqrt(2.0 / n_slots), var
    assert float(resid.min()) > 0.85 and float(resid.max()) < 1.15
    v = torch.cat([w.prefix_value, w.new_value]).float()
    assert abs(float(v.mean(dim=0).var())) < 0.01        # values carry no bias


def test_outlier_channels_are_one_percent_scaled_by_eight():
    spec = inputs.CHUNKED_PREFILL.replace(name="outlier_check", n_prefill=2, prefill_qlen=256,
                                          prefix_lens=(1000, 1200))
    w = inputs.make_workload(spec)
    k = _all_keys(w).reshape(-1, spec.hk * spec.d)
    std = k.std(dim=0)
    big = std > 4.0
    assert int(big.sum()) == round(0.01 * spec.hk * spec.d) == 10
    assert float(std[big].min()) > 7.0 and float(std[big].max()) < 9.0
    assert float(std[~big].max()) < 1.2

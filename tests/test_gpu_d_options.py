"""GPU parity of the attention options against the CPU oracle: the
non-causal mode (the first pass of attention over a cached prefix), the prefix
pass merged with the new keys, attention sinks, sliding windows, the q-range
status bit and the test hook that makes the pipeline waits run out.

The oracle sees only the generated host inputs; its options are pinned in
tests/test_oracle_pins.py."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_attention_int8_gb300 import _lib, inputs
from tests import _harness as H

pytestmark = pytest.mark.gpu

SQRT2 = math.sqrt(2.0)

SPECS = {
    # single-token rows: the decode kernel (split and unsplit)
    "decode": inputs.Spec("opt_decode", 301, hq=32, hk=8, d=128, bs=16, n_decode=5,
                          decode_lens=(90, 700), k_bias_std=SQRT2),
    # multi-token chunks on cached prefixes: the tcgen05 prefill kernel
    "prefill": inputs.Spec("opt_prefill", 302, hq=32, hk=8, d=128, bs=16, n_prefill=3,
                           prefill_qlen=150, prefix_lens=(0, 300), k_outlier_frac=0.01),
    # prefill chunks and decodes in one batch, block size 32
    "mixed": inputs.Spec("opt_mixed", 303, hq=64, hk=8, d=128, bs=32, n_prefill=2,
                         prefill_qlen=70, prefix_lens=(0, 130), n_decode=4,
                         decode_lens=(40, 400), pad_frac=0.05),
    # D = 256 chunks: the generic mma.sync kernel
    "d256": inputs.Spec("opt_d256", 304, hq=16, hk=4, d=256, bs=32, n_prefill=2,
                        prefill_qlen=45, prefix_lens=(10, 120), n_decode=2,
                        decode_lens=(30, 300)),
    # 16 q heads per kv head: the generic kernel takes every row, split ones too
    "qpk16": inputs.Spec("opt_qpk16", 305, hq=16, hk=1, d=128, bs=16, n_prefill=1,
                         prefill_qlen=33, prefix_lens=(5, 60), n_decode=3,
                         decode_lens=(20, 300)),
    # D = 64 on the tcgen05 kernel
    "d64": inputs.Spec("opt_d64", 306, hq=8, hk=2, d=64, bs=16, n_prefill=2,
                       prefill_qlen=300, prefix_lens=(0, 90), n_decode=2, decode_lens=(5, 90)),
}

_state_cache = {}


def _states(name, device):
    if name not in _state_cache:
        w = inputs.make_workload(SPECS[name])
        _state_cache[name] = (H.GpuState(w, device), H.OracleState(w))
    return _state_cache[name]


def _sinks(hq, kind, seed=0):
    """Sink logits per q head: a mix of -inf (no sink), 0, 30 and random values."""
    if kind is None:
        return None
    rng = np.random.default_rng(seed)
    if kind == "mix":
        pool = np.array([-np.inf, 0.0, 30.0, 1.5, -2.0], np.float32)
        s = pool[np.arange(hq) % pool.size].copy()
        s[4::5] = rng.standard_normal(s[4::5].size) * 3.0
        return s.astype(np.float32)
    return np.full(hq, float(kind), np.float32)


def _gpu(g, num_splits=None, seq_lens=None, block_table=None, **kw):
    w = g.w
    ns = w.spec.num_splits if num_splits is None else num_splits
    sl = g.seq_lens if seq_lens is None else seq_lens.to(g.device)
    bt = g.block_table if block_table is None else block_table.to(g.device)
    ws = torch.zeros(_lib.workspace_size(w.num_seqs, w.spec.hq, w.spec.d, ns),
                     dtype=torch.uint8, device=g.device)
    out = torch.full_like(g.q, float("nan"))
    lse = torch.full((w.num_tokens, w.spec.hq), float("nan"), device=g.device)
    sinks = kw.pop("sinks", None)
    if sinks is not None:
        sinks = torch.from_numpy(sinks).to(g.device)
    max_seq_len = kw.pop("max_seq_len", None) or max(1, int(sl.max().item()))
    _lib.paged_attention(g.q, g.kc, g.ks, g.vc, g.vs, g.cu, sl, bt, w.max_query_len,
                         max_seq_len, w.softmax_scale, num_splits=ns, out=out, lse=lse,
                         workspace=ws, sinks=sinks, **kw)
    assert _lib.check_status(ws) == 0
    return out, lse


def _oracle(o, rows, seq_lens=None, block_table=None, **kw):
    w = o.w
    sl = w.seq_lens if seq_lens is None else seq_lens
    bt = w.block_table if block_table is None else block_table
    return oracle.paged_attention(inputs.bf16_bits(w.q), o.kc, o.ks, o.vc, o.vs,
                                  w.cu_seqlens_q.numpy(), sl.numpy(), bt.numpy(),
                                  w.softmax_scale, rows=rows, **kw)


def _compare(out, lse, ref_out, ref_lse, rows, label, single_key=False):
    """Element-wise comparison where LSEs may be -inf (rows with no key and no
    sink): those rows must be -inf on both sides with out exactly 0.

    single_key: every row sees exactly one key, so its output is that key's
    dequantized V row, rounded to the bf16 output format (through the fp16 V
    operand).  That rounding alone has a mean error of about 1.02e-3 on N(0,1)
    values, and half a bf16 step is 0.0156 for values in [4, 8): more than
    the 1e-3 mean and 1e-2 max bounds, which hold for averaged outputs.  Here
    the max bound is widened by one bf16 step of the value (2^-7 |v|), and the
    mean bound is taken against the oracle's output rounded to bf16."""
    d = out.shape[-1]
    o = out.float().cpu().numpy().reshape(-1, d)[rows].astype(np.float64)
    lg = lse.cpu().numpy().reshape(-1)[rows].astype(np.float64)
    empty = np.isneginf(ref_lse)
    assert np.all(np.isneginf(lg[empty])), f"{label}: empty rows need lse = -inf"
    assert np.all(o[empty] == 0.0), f"{label}: empty rows need out = 0"
    full = ~empty
    if not np.any(full):
        return
    if single_key:
        ref = ref_out[full]
        assert np.all(np.abs(o[full] - ref) <= H.OUT_MAX + 2.0 ** -7 * np.abs(ref)), label
        ref_bf = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        assert np.mean(np.abs(o[full] - ref_bf)) <= H.OUT_MEAN, label
        lg = lse.cpu().numpy().reshape(-1)[rows[full]].astype(np.float64)
        rel = np.abs(lg - ref_lse[full]) / np.maximum(1.0, np.abs(ref_lse[full]))
        assert rel.max() <= H.LSE_REL, label
        return
    H.compare(out, lse, ref_out[full], ref_lse[full], rows[full], label=label)


# ----------------------------------------------------------------------------- non-causal


@pytest.mark.parametrize("name", ["prefill", "mixed", "d256", "qpk16", "d64", "decode"])
def test_non_causal_matches_oracle(name, cuda_device):
    # every query sees all seq_len keys; seq_len taken below, at and above
    # q_len, and 0 (rows with no key: out = 0, lse = -inf)
    g, o = _states(name, cuda_device)
    w = g.w
    ql = w.q_lens.numpy()
    L = w.seq_lens.numpy().copy()
    sl = L.copy()
    sl[0] = 0
    if w.num_seqs > 1:
        sl[1] = max(0, int(ql[1]) // 2)
    if w.num_seqs > 2:
        sl[2] = max(0, int(L[2]) - 7)
    sl_t = torch.from_numpy(sl.astype(np.int32))
    rows = H.owned_rows(w)
    ref_out, ref_lse = _oracle(o, rows, seq_lens=sl_t, causal=False)
    splits = (None, 4) if w.max_query_len == 1 or name in ("mixed", "qpk16", "d256") else (None,)
    for ns in splits:
        out, lse = _gpu(g, num_splits=ns, seq_lens=sl_t, causal=False,
                        max_seq_len=int(L.max()))
        _compare(out, lse, ref_out, ref_lse, rows, f"{name} non-causal splits={ns}")


@pytest.mark.parametrize("bs,d,hq,hk", [(16, 128, 32, 8), (32, 64, 8, 2), (16, 256, 16, 4),
                                        (32, 128, 16, 1)])
def test_prefix_pass_merged_with_new_keys_equals_one_causal_pass(bs, d, hq, hk, cuda_device):
    """Attention over a cached prefix plus new keys in two passes, as the
    page's `_attend_with_prefix` does it: the prefix non-causally, the new keys
    causally (block table shifted past the prefix pages), merged by LSE with
    merge_attn_states -- against the oracle's single causal pass."""
    spec = inputs.Spec(f"prefix_{bs}_{d}", 310 + d + bs, hq=hq, hk=hk, d=d, bs=bs,
                       prefill_qlen=70, fixed_prefix_lens=(0, bs, 3 * bs, 7 * bs))
    w = inputs.make_workload(spec)
    g, o = H.GpuState(w, cuda_device), H.OracleState(w)
    ql = w.q_lens.numpy()
    prefix = w.seq_lens.numpy() - ql
    assert np.all(prefix % bs == 0)
    rows = H.owned_rows(w)
    ref_out, ref_lse = o.attention(rows=rows)
    # pass 1: the prefix, every query sees all of it
    out_a, lse_a = _gpu(g, seq_lens=torch.from_numpy(prefix.astype(np.int32)), causal=False,
                        max_seq_len=int(w.seq_lens.max()))
    # pass 2: the new keys only, causal, through the pages after the prefix
    bt = w.block_table.numpy()
    bt2 = np.full_like(bt, -1)
    for s in range(w.num_seqs):
        n = bt.shape[1] - prefix[s] // bs
        bt2[s, :n] = bt[s, prefix[s] // bs:]
    out_b, lse_b = _gpu(g, seq_lens=torch.from_numpy(ql.astype(np.int32)),
                        block_table=torch.from_numpy(bt2), max_seq_len=int(ql.max()))
    out, lse = _lib.merge_attn_states(out_a, lse_a, out_b, lse_b)
    H.compare(out, lse, ref_out, ref_lse, rows, label=f"prefix pass bs={bs} d={d}")


# ----------------------------------------------------------------------------- sinks, window


OPTION_CASES = [
    # (sliding window, sinks)
    (0, "mix"),
    (1, None),
    (16, "mix"),
    (37, None),
    (37, 30.0),
    (100000, "-inf"),
]


@pytest.mark.parametrize("window,sinks", OPTION_CASES)
@pytest.mark.parametrize("name", ["decode", "prefill", "mixed", "d256", "qpk16", "d64"])
def test_sinks_and_sliding_window_match_oracle(name, window, sinks, cuda_device):
    g, o = _states(name, cuda_device)
    w = g.w
    sk = _sinks(w.spec.hq, float("-inf") if sinks == "-inf" else sinks, seed=window)
    rows = H.owned_rows(w)
    ref_out, ref_lse = _oracle(o, rows, sinks=sk, window=window)
    splits = (None, 1, 3, 16) if name in ("decode", "qpk16") else (None, 4)
    for ns in splits:
        out, lse = _gpu(g, num_splits=ns, sinks=sk, sliding_window=window)
        _compare(out, lse, ref_out, ref_lse, rows,
                 f"{name} window={window} sinks={sinks} splits={ns}",
                 single_key=window == 1 and sinks is None)


def test_window_splits_follow_the_window_not_the_hint(cuda_device):
    # long decode rows with a short window: only the window's tiles are split
    spec = inputs.Spec("win_long", 320, hq=32, hk=8, d=128, bs=16,
                       fixed_decode_lens=(5000, 4100, 64, 1), k_bias_std=SQRT2)
    w = inputs.make_workload(spec)
    g, o = H.GpuState(w, cuda_device), H.OracleState(w)
    rows = H.owned_rows(w)
    for window in (100, 1000, 4097):
        ref_out, ref_lse = _oracle(o, rows, window=window)
        for ns in (0, 2, 16):
            out, lse = _gpu(g, num_splits=ns, sliding_window=window)
            _compare(out, lse, ref_out, ref_lse, rows, f"window={window} splits={ns}")


def test_window_never_reads_pages_before_it(cuda_device):
    # block-table entries of pages wholly before every query's window are
    # garbage (freed pages): the result and the status word do not change
    spec = inputs.Spec("win_pages", 321, hq=32, hk=8, d=128, bs=16, n_prefill=2,
                       prefill_qlen=64, fixed_prefix_lens=(320, 640), n_decode=0)
    w = inputs.make_workload(spec)
    g, o = H.GpuState(w, cuda_device), H.OracleState(w)
    rows = H.owned_rows(w)
    window = 48
    ref_out, ref_lse = _oracle(o, rows, window=window)
    bt = w.block_table.clone()
    prefix = (w.seq_lens - w.q_lens).numpy()
    for s in range(w.num_seqs):
        dead = (prefix[s] - window) // 16  # pages every query of the chunk is past
        bt[s, :max(dead, 0)] = 1 << 30
    out, lse = _gpu(g, sliding_window=window, block_table=bt)
    _compare(out, lse, ref_out, ref_lse, rows, "window with stale pages")


# ----------------------------------------------------------------------------- status bits


@pytest.mark.parametrize("name", ["decode", "prefill", "d256"])
def test_q_beyond_fp16_range_is_flagged(name, cuda_device):
    g, o = _states(name, cuda_device)
    w = g.w
    q_bad = g.q.clone()
    q_bad[0, 0, 5] = 1.0e5  # rounds to inf in fp16 (first token: a prefill chunk, if any)
    q_bad[-1, 1, 7] = -1.0e5  # last token: a decode row, if any
    ws = torch.zeros(_lib.workspace_size(w.num_seqs, w.spec.hq, w.spec.d, 1), dtype=torch.uint8,
                     device=cuda_device)
    _lib.paged_attention(q_bad, g.kc, g.ks, g.vc, g.vs, g.cu, g.seq_lens, g.block_table,
                         w.max_query_len, w.max_seq_len, num_splits=1, workspace=ws)
    with pytest.raises(_lib.PagedAttentionError) as e:
        _lib.check_status(ws)
    assert e.value.bits == _lib.DEV_BAD_Q
    assert e.value.status == _lib.Status.DEVICE_CHECK
    # a large bf16 value that stays finite in fp16 (65280 = 255 * 2^8) is not flagged
    q_ok = g.q.clone()
    q_ok[0, 0, 5] = 65280.0
    q_ok[-1, 1, 7] = -65280.0
    _lib.paged_attention(q_ok, g.kc, g.ks, g.vc, g.vs, g.cu, g.seq_lens, g.block_table,
                         w.max_query_len, w.max_seq_len, num_splits=1, workspace=ws)
    assert _lib.check_status(ws) == 0


def test_wait_timeout_is_reported_and_the_context_stays_usable(cuda_device):
    # the test hook stages nothing: every consumer wait of the decode kernel
    # gives up after ~1 ms, the call reports PA_ERR_TIMEOUT, and a clean call on
    # the same context afterwards still matches the oracle
    g, o = _states("decode", cuda_device)
    w = g.w
    for ns in (1, 4):
        ws = torch.zeros(_lib.workspace_size(w.num_seqs, w.spec.hq, w.spec.d, ns),
                         dtype=torch.uint8, device=cuda_device)
        _lib.paged_attention(g.q, g.kc, g.ks, g.vc, g.vs, g.cu, g.seq_lens, g.block_table, 1,
                             w.max_seq_len, num_splits=ns, workspace=ws,
                             flags=_lib.ATTN_TEST_TIMEOUT)
        with pytest.raises(_lib.PagedAttentionError) as e:
            _lib.check_status(ws)
        assert e.value.status == _lib.Status.TIMEOUT
        assert e.value.bits & _lib.DEV_TIMEOUT
    rows = H.owned_rows(w)
    ref_out, ref_lse = o.attention(rows=rows)
    for ns in (1, 4):
        out, lse = _gpu(g, num_splits=ns)
        H.compare(out, lse, ref_out, ref_lse, rows, label=f"after timeout splits={ns}")

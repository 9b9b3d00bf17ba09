"""GPU parity of the alternative cache format -- fp8 (e4m3) keys and 4-bit
values with one fp16 scale and zero per key -- against the CPU oracle: the
store bit for bit (codes, nibbles, scales, zeros and placement, for tokens
that share a nibble byte within one call and for tokens whose byte mate is
already in the cache), then attention over that cache element by element --
decode rows (the decode kernel of the format) and prefill chunks and rows of
16 q heads per kv head (the generic kernel in the format), split and
unsplit, with sinks, a sliding window and the non-causal prefix pass."""
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
    "decode": inputs.Spec("f8_decode", 501, hq=32, hk=8, d=128, bs=16, n_decode=6,
                          decode_lens=(100, 900), k_bias_std=SQRT2),
    "d256": inputs.Spec("f8_d256", 502, hq=16, hk=4, d=256, bs=32, n_decode=4,
                        decode_lens=(40, 700), k_bias_std=SQRT2),
    "d64": inputs.Spec("f8_d64", 503, hq=8, hk=2, d=64, bs=16, n_decode=5,
                       decode_lens=(1, 300)),
    "long": inputs.Spec("f8_long", 504, hq=32, hk=8, d=128, bs=32,
                        fixed_decode_lens=(3000, 2111, 17), k_bias_std=SQRT2, num_splits=16),
    # prefill chunks (the generic kernel in this format) beside decode rows
    "prefill": inputs.Spec("f8_prefill", 506, hq=32, hk=8, d=128, bs=16, n_prefill=3,
                           prefill_qlen=150, prefix_lens=(0, 400), n_decode=3,
                           decode_lens=(50, 700), k_bias_std=SQRT2),
    "prefill_d256": inputs.Spec("f8_prefill_d256", 507, hq=16, hk=4, d=256, bs=32, n_prefill=2,
                                prefill_qlen=70, prefix_lens=(0, 200), n_decode=2,
                                decode_lens=(30, 300)),
    "prefill_d64": inputs.Spec("f8_prefill_d64", 508, hq=8, hk=2, d=64, bs=16, n_prefill=2,
                               prefill_qlen=100, prefix_lens=(0, 150), n_decode=2,
                               decode_lens=(1, 200)),
    # 16 q heads per kv head: every row, decode rows included, in the generic kernel
    "wide": inputs.Spec("f8_wide", 509, hq=32, hk=2, d=128, bs=16, n_prefill=2,
                        prefill_qlen=40, prefix_lens=(0, 300), n_decode=4,
                        decode_lens=(20, 900)),
}


class F8State:
    """The workload stored in the fp8 / 4-bit format on the GPU (by the
    library) and on the host (by the oracle), from the same generated rows."""

    def __init__(self, w, device, batches=None):
        s = w.spec
        self.w, self.device = w, device
        self.kc, self.vc, self.vs, self.vz = inputs.empty_cache_f8v4(w.num_blocks, s.hk, s.bs, s.d,
                                                                     device=device)
        okc, ovc, ovs, ovz = inputs.empty_cache_f8v4(w.num_blocks, s.hk, s.bs, s.d)
        self.okc, self.ovc = okc.numpy(), ovc.numpy()
        self.ovs, self.ovz = ovs.numpy().view(np.uint16), ovz.numpy().view(np.uint16)
        status = torch.zeros(4, dtype=torch.int32, device=device)
        if batches is None:
            batches = [(w.prefix_key, w.prefix_value, w.prefix_slots),
                       (w.new_key, w.new_value, w.new_slots)]
        for k, v, sl in batches:
            if k.shape[0] == 0:
                continue
            _lib.kv_store_f8v4(k.to(device), v.to(device), sl.to(device), self.kc, self.vc,
                               self.vs, self.vz, status=status)
            assert oracle.kv_store_f8v4(inputs.bf16_bits(k), inputs.bf16_bits(v), sl.numpy(),
                                        self.okc, self.ovc, self.ovs, self.ovz) == 0
        assert _lib.check_status(status) == 0
        self.q = w.q.to(device)
        self.cu = w.cu_seqlens_q.to(device)
        self.seq_lens = w.seq_lens.to(device)
        self.bt = w.block_table.to(device)

    def assert_cache_equal(self):
        np.testing.assert_array_equal(self.kc.cpu().numpy(), self.okc)
        np.testing.assert_array_equal(self.vc.cpu().numpy(), self.ovc)
        np.testing.assert_array_equal(self.vs.cpu().numpy().view(np.uint16), self.ovs)
        np.testing.assert_array_equal(self.vz.cpu().numpy().view(np.uint16), self.ovz)

    def gpu(self, num_splits=0, sinks=None, window=0, causal=True):
        w = self.w
        ws = torch.zeros(_lib.workspace_size(w.num_seqs, w.spec.hq, w.spec.d, num_splits),
                         dtype=torch.uint8, device=self.device)
        out = torch.full_like(self.q, float("nan"))
        lse = torch.full((w.num_tokens, w.spec.hq), float("nan"), device=self.device)
        sk = None if sinks is None else torch.from_numpy(sinks).to(self.device)
        _lib.paged_attention_f8v4(self.q, self.kc, self.vc, self.vs, self.vz, self.cu,
                                  self.seq_lens, self.bt, w.max_query_len, w.max_seq_len,
                                  w.softmax_scale, num_splits=num_splits, out=out, lse=lse,
                                  workspace=ws, sinks=sk, sliding_window=window, causal=causal)
        assert _lib.check_status(ws) == 0
        return out, lse

    def oracle(self, rows, sinks=None, window=0, causal=True):
        w = self.w
        return oracle.paged_attention(inputs.bf16_bits(w.q), self.okc, None, self.ovc, self.ovs,
                                      w.cu_seqlens_q.numpy(), w.seq_lens.numpy(),
                                      w.block_table.numpy(), w.softmax_scale, rows=rows,
                                      sinks=sinks, window=window, causal=causal,
                                      v_zero=self.ovz)


_cache = {}


def _state(name, device):
    if name not in _cache:
        _cache[name] = F8State(inputs.make_workload(SPECS[name]), device)
    return _cache[name]


@pytest.mark.parametrize("name", sorted(SPECS))
def test_f8v4_store_is_bit_exact(name, cuda_device):
    _state(name, cuda_device).assert_cache_equal()


def test_f8v4_store_keeps_byte_mates_from_earlier_calls(cuda_device):
    # one token per call (decode steps): each token's nibble byte is shared
    # with a token stored by an earlier call, and both must survive
    spec = inputs.Spec("f8_steps", 505, hq=8, hk=2, d=64, bs=16, fixed_decode_lens=(40,))
    w = inputs.make_workload(spec)
    k, v, sl = w.all_key_value()
    order = np.random.default_rng(0).permutation(k.shape[0])
    batches = [(k[i:i + 1], v[i:i + 1], sl[i:i + 1]) for i in order]
    F8State(w, cuda_device, batches=batches).assert_cache_equal()


@pytest.mark.parametrize("name", sorted(SPECS))
def test_f8v4_attention_matches_oracle(name, cuda_device):
    g = _state(name, cuda_device)
    rows = H.owned_rows(g.w)
    ref_out, ref_lse = g.oracle(rows)
    for ns in (1, 4, 0):
        out, lse = g.gpu(num_splits=ns)
        H.compare(out, lse, ref_out, ref_lse, rows, label=f"f8v4 {name} splits={ns}")


@pytest.mark.parametrize("window,sink", [(37, 1.5), (1000, None), (0, -2.0)])
def test_f8v4_sinks_and_window(window, sink, cuda_device):
    g = _state("decode", cuda_device)
    rows = H.owned_rows(g.w)
    sinks = None if sink is None else np.full(g.w.spec.hq, sink, np.float32)
    ref_out, ref_lse = g.oracle(rows, sinks=sinks, window=window)
    for ns in (1, 3):
        out, lse = g.gpu(num_splits=ns, sinks=sinks, window=window)
        H.compare(out, lse, ref_out, ref_lse, rows, label=f"f8v4 window={window} sink={sink}")


@pytest.mark.parametrize("window,sink,causal", [(60, 1.0, True), (0, None, False),
                                                (0, -1.0, False), (500, None, True)])
def test_f8v4_prefill_options(window, sink, causal, cuda_device):
    g = _state("prefill", cuda_device)
    rows = H.owned_rows(g.w)
    sinks = None if sink is None else np.full(g.w.spec.hq, sink, np.float32)
    ref_out, ref_lse = g.oracle(rows, sinks=sinks, window=window, causal=causal)
    for ns in (1, 4):
        out, lse = g.gpu(num_splits=ns, sinks=sinks, window=window, causal=causal)
        H.compare(out, lse, ref_out, ref_lse, rows,
                  label=f"f8v4 prefill window={window} sink={sink} causal={causal} splits={ns}")


@pytest.mark.parametrize("d,bs", [(64, 16), (128, 32), (256, 16)])
def test_f8v4_store_padding_bad_slots_and_strided_rows(d, bs, cuda_device):
    # padding rows, two slots past the cache (flagged, skipped for K and V),
    # a run of consecutive slots then a shuffled tail, and key / value rows
    # with a token stride past hk * D (16-byte aligned)
    rng = np.random.default_rng(510 + d + bs)
    n, hk, pad = 203, 3, 8
    num_blocks = (n + bs - 1) // bs + 4
    nslots = num_blocks * bs
    slots = np.arange(n, dtype=np.int64)
    tail = n // 3
    slots[-tail:] = rng.permutation(np.arange(n - tail, nslots))[:tail]
    slots[rng.choice(n, size=9, replace=False)] = -1
    bad = rng.choice(np.flatnonzero(slots >= 0), size=2, replace=False)
    slots[bad] = [nslots, nslots + 77]
    rows = [torch.from_numpy(rng.standard_normal((n, hk * d + pad)) * 3.0).to(torch.bfloat16)
            for _ in range(2)]
    k, v = (r[:, :hk * d].reshape(n, hk, d) for r in rows)
    kc, vc, vs, vz = inputs.empty_cache_f8v4(num_blocks, hk, bs, d, device=cuda_device)
    status = torch.zeros(4, dtype=torch.int32, device=cuda_device)
    kd, vd = (r.to(cuda_device).as_strided((n, hk, d), (hk * d + pad, d, 1)) for r in rows)
    _lib.kv_store_f8v4(kd, vd, torch.from_numpy(slots).to(cuda_device), kc, vc, vs, vz,
                       status=status)
    okc, ovc, ovs, ovz = inputs.empty_cache_f8v4(num_blocks, hk, bs, d)
    okc, ovc = okc.numpy(), ovc.numpy()
    ovs, ovz = ovs.numpy().view(np.uint16), ovz.numpy().view(np.uint16)
    assert oracle.kv_store_f8v4(inputs.bf16_bits(k.contiguous()), inputs.bf16_bits(v.contiguous()),
                                slots, okc, ovc, ovs, ovz) == 2
    with pytest.raises(_lib.PagedAttentionError) as e:
        _lib.check_status(status)
    assert e.value.bits == _lib.DEV_BAD_SLOT
    np.testing.assert_array_equal(kc.cpu().numpy(), okc)
    np.testing.assert_array_equal(vc.cpu().numpy(), ovc)
    np.testing.assert_array_equal(vs.cpu().numpy().view(np.uint16), ovs)
    np.testing.assert_array_equal(vz.cpu().numpy().view(np.uint16), ovz)

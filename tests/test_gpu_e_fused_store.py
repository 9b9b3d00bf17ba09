"""GPU parity of the fused RMSNorm + rotation q8 store (kv_store_norm_rope)
against the CPU oracle: the whole cache -- codes, scales and placement --
bit for bit, for every head size and block size, split-half and interleaved
pairs, full and partial rotation, with and without the norm, padding rows
and positions outside the table; then attention over a cache filled this way
against the oracle's attention over the oracle's cache."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_attention_int8_gb300 import _lib, inputs
from tests import _harness as H

pytestmark = pytest.mark.gpu


def _rope_table(max_pos, pairs, base=10000.0):
    """cos / sin of position p and pair i at the angle p * base^(-2i / (2 pairs)),
    the usual rotary frequencies, as fp32 [max_pos, pairs, 2]."""
    inv_freq = base ** (-np.arange(pairs, dtype=np.float64) / pairs)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], -1).astype(np.float32)


def _case(seed, hk, d, bs, n, rot, interleaved, norm, bad_pos=False, outliers=False):
    rng = np.random.default_rng(seed)
    num_blocks = (n + bs - 1) // bs + 3
    # consecutive slots in page order (whole pages, prefill-like) then a
    # shuffled tail (decode-like), and padding rows
    slots = np.arange(n, dtype=np.int64)
    tail = n // 3
    slots[-tail:] = rng.permutation(np.arange(n - tail, num_blocks * bs))[:tail]
    slots[rng.choice(n, size=max(1, n // 25), replace=False)] = -1
    max_pos = 4096
    positions = rng.integers(0, max_pos, n).astype(np.int64)
    if bad_pos:
        positions[rng.choice(n, size=3, replace=False)] = [max_pos, -1, max_pos + 7]
    k = rng.standard_normal((n, hk, d)) * 2.0
    if outliers:
        k[:, :, rng.choice(d, size=3, replace=False)] *= 8.0
    k = torch.from_numpy(k).to(torch.bfloat16)
    v = torch.from_numpy(rng.standard_normal((n, hk, d))).to(torch.bfloat16)
    w = torch.from_numpy(rng.uniform(0.3, 1.7, d)).to(torch.bfloat16) if norm else None
    table = _rope_table(max_pos, rot // 2) if rot else None
    return dict(k=k, v=v, slots=slots, positions=positions, w=w, table=table,
                num_blocks=num_blocks, hk=hk, d=d, bs=bs, interleaved=interleaved)


def _strided_key(k, device, pad):
    """k [n, hk, d] on the device with a token stride of hk * d + pad
    elements (pad = 1: rows that are not 16-byte aligned)."""
    n, hk, d = k.shape
    if pad == 0:
        return k.to(device)
    big = torch.zeros((n, hk * d + pad), dtype=k.dtype, device=device)
    big[:, :hk * d] = k.reshape(n, hk * d).to(device)
    return big.as_strided((n, hk, d), (hk * d + pad, d, 1))


def _run_both(c, device, eps=1e-6, key_pad=0):
    kc, ks, vc, vs = inputs.empty_cache(c["num_blocks"], c["hk"], c["bs"], c["d"], device=device)
    status = torch.zeros(4, dtype=torch.int32, device=device)
    table = None if c["table"] is None else torch.from_numpy(c["table"]).to(device)
    _lib.kv_store_norm_rope(_strided_key(c["k"], device, key_pad), c["v"].to(device),
                            torch.from_numpy(c["slots"]).to(device), kc, ks, vc, vs,
                            positions=torch.from_numpy(c["positions"]).to(device),
                            norm_weight=None if c["w"] is None else c["w"].to(device), eps=eps,
                            rope=table, interleaved=c["interleaved"], status=status)
    # copies taken on the same stream right after the call: the store's work
    # on any other stream has joined it by then
    kc, ks, vc, vs = (t.clone() for t in (kc, ks, vc, vs))
    torch.cuda.synchronize()
    okc, oks, ovc, ovs = [t.numpy() for t in inputs.empty_cache(c["num_blocks"], c["hk"],
                                                                c["bs"], c["d"])]
    oks, ovs = oks.view(np.uint16), ovs.view(np.uint16)
    bad = oracle.kv_store_norm_rope(inputs.bf16_bits(c["k"]), inputs.bf16_bits(c["v"]),
                                    c["slots"], c["positions"], okc, oks, ovc, ovs,
                                    None if c["w"] is None else inputs.bf16_bits(c["w"]), eps,
                                    c["table"], interleaved=c["interleaved"])
    return (kc, ks, vc, vs, status), (okc, oks, ovc, ovs, bad)


def _assert_same(g, o):
    kc, ks, vc, vs, _ = g
    okc, oks, ovc, ovs, _ = o
    np.testing.assert_array_equal(kc.cpu().numpy(), okc)
    np.testing.assert_array_equal(ks.cpu().numpy().view(np.uint16), oks)
    np.testing.assert_array_equal(vc.cpu().numpy(), ovc)
    np.testing.assert_array_equal(vs.cpu().numpy().view(np.uint16), ovs)


@pytest.mark.parametrize("d,bs,rot,interleaved,norm", [
    (128, 16, 128, False, True),
    (128, 16, 128, True, True),
    (128, 32, 64, False, True),    # partial rotation: channels 64.. pass through
    (128, 16, 96, True, False),    # rotation only, a rotary dim not a multiple of 32
    (64, 16, 64, False, True),
    (64, 32, 32, True, True),
    (256, 16, 256, False, True),
    (256, 32, 128, True, True),
    (128, 16, 0, False, True),     # norm only
])
def test_fused_store_is_bit_exact(d, bs, rot, interleaved, norm, cuda_device):
    c = _case(400 + d + rot + bs + int(interleaved), hk=3, d=d, bs=bs, n=157, rot=rot,
              interleaved=interleaved, norm=norm, outliers=True)
    for key_pad in (0, 1):  # key rows 16-byte aligned or not
        g, o = _run_both(c, cuda_device, key_pad=key_pad)
        assert o[4] == 0
        assert _lib.check_status(g[4]) == 0
        _assert_same(g, o)


@pytest.mark.parametrize("d,rot,interleaved,key_pad", [
    (128, 128, False, 0), (128, 128, True, 0), (256, 192, False, 0), (64, 64, False, 0),
    (128, 128, False, 1), (256, 256, True, 1)])
def test_fused_store_large_batch_is_bit_exact(d, rot, interleaved, key_pad, cuda_device):
    # enough tokens for one warp per token walking the kv heads (the
    # population / prefill launch shape) rather than one per (token, head),
    # and the values beside them on a second stream; key_pad 1: key rows
    # that are not 16-byte aligned
    c = _case(430 + d + rot + int(interleaved), hk=2, d=d, bs=16, n=40000, rot=rot,
              interleaved=interleaved, norm=True, outliers=True)
    g, o = _run_both(c, cuda_device, key_pad=key_pad)
    assert o[4] == 0
    assert _lib.check_status(g[4]) == 0
    _assert_same(g, o)


def test_fused_store_without_norm_or_rotation_equals_kv_store(cuda_device):
    c = _case(410, hk=2, d=128, bs=16, n=100, rot=0, interleaved=False, norm=False)
    g, _ = _run_both(c, cuda_device)
    kc, ks, vc, vs = inputs.empty_cache(c["num_blocks"], 2, 16, 128, device=cuda_device)
    _lib.kv_store(c["k"].to(cuda_device), c["v"].to(cuda_device),
                  torch.from_numpy(c["slots"]).to(cuda_device), kc, ks, vc, vs)
    for a, b in zip(g[:4], (kc, ks, vc, vs)):
        assert torch.equal(a, b)


def test_positions_outside_the_table_are_flagged_and_skipped(cuda_device):
    c = _case(411, hk=2, d=128, bs=16, n=90, rot=128, interleaved=False, norm=True, bad_pos=True)
    for key_pad in (0, 1):
        g, o = _run_both(c, cuda_device, key_pad=key_pad)
        assert o[4] >= 1
        with pytest.raises(_lib.PagedAttentionError) as e:
            _lib.check_status(g[4])
        assert e.value.bits == _lib.DEV_BAD_POS
        _assert_same(g, o)


def test_slots_outside_the_cache_are_flagged_and_skipped(cuda_device):
    c = _case(412, hk=2, d=128, bs=16, n=90, rot=128, interleaved=True, norm=True)
    nslots = c["num_blocks"] * c["bs"]
    c["slots"][[5, 40]] = [nslots, nslots + 100]
    for key_pad in (0, 1):
        g, o = _run_both(c, cuda_device, key_pad=key_pad)
        assert o[4] == 2
        with pytest.raises(_lib.PagedAttentionError) as e:
            _lib.check_status(g[4])
        assert e.value.bits == _lib.DEV_BAD_SLOT
        _assert_same(g, o)


def test_attention_over_a_fused_store_cache(cuda_device):
    # a small chunked-prefill batch stored with norm + rotation (positions =
    # the tokens' places in their sequences), attended on the GPU and by the
    # oracle over its own fused-store cache
    spec = inputs.Spec("fused_attn", 420, hq=32, hk=8, d=128, bs=16, n_prefill=3,
                       prefill_qlen=90, prefix_lens=(0, 200), n_decode=3,
                       decode_lens=(30, 300))
    w = inputs.make_workload(spec)
    k, v, slots = w.all_key_value()
    # position of every stored row: its index within its sequence
    L = w.seq_lens.numpy()
    ql = w.q_lens.numpy()
    pos_prefix = np.concatenate([np.arange(L[s] - ql[s]) for s in range(w.num_seqs)])
    pos_new = np.concatenate([np.arange(L[s] - ql[s], L[s]) for s in range(w.num_seqs)])
    positions = np.concatenate([pos_prefix, pos_new]).astype(np.int64)
    table = _rope_table(int(L.max()) + 1, 64)
    wt = torch.from_numpy(np.random.default_rng(3).uniform(0.5, 1.5, 128)).to(torch.bfloat16)
    dev = cuda_device
    g = H.GpuState(w, dev, populate=False)
    _lib.kv_store_norm_rope(k.to(dev), v.to(dev), slots.to(dev), g.kc, g.ks, g.vc, g.vs,
                            positions=torch.from_numpy(positions).to(dev), norm_weight=wt.to(dev),
                            rope=torch.from_numpy(table).to(dev), status=g.status)
    assert _lib.check_status(g.status) == 0
    o = H.OracleState.__new__(H.OracleState)
    o.w = w
    kc, ks, vc, vs = inputs.empty_cache(w.num_blocks, 8, 16, 128)
    o.kc, o.vc = kc.numpy(), vc.numpy()
    o.ks, o.vs = ks.numpy().view(np.uint16), vs.numpy().view(np.uint16)
    assert oracle.kv_store_norm_rope(inputs.bf16_bits(k), inputs.bf16_bits(v), slots.numpy(),
                                     positions, o.kc, o.ks, o.vc, o.vs, inputs.bf16_bits(wt),
                                     1e-6, table) == 0
    H.assert_cache_equal(g, o)
    rows = H.owned_rows(w)
    ref_out, ref_lse = o.attention(rows=rows)
    out, lse = g.attention()
    H.compare(out, lse, ref_out, ref_lse, rows, label="attention over the fused store")

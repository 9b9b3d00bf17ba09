"""GPU parity of pa_merge_attn_states (the log-sum-exp merge `_merge_lse_` of
"shared/attention_kit.py", natural-log LSE) against the oracle's
merge_states, and the two-pass identity it serves: a decode row attended over
its sequence's first P keys and, through a block table shifted by P / bs
pages, over the remaining keys, merged by LSE, equals one pass over all keys."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_attention_int8_gb300 import _lib, inputs
from tests import _harness as H

pytestmark = pytest.mark.gpu

SQRT2 = math.sqrt(2.0)


def _states(rng, rows, d):
    a = torch.from_numpy(rng.standard_normal((rows, d)).astype(np.float32)).to(torch.bfloat16)
    b = torch.from_numpy(rng.standard_normal((rows, d)).astype(np.float32)).to(torch.bfloat16)
    la = rng.uniform(-5.0, 20.0, rows).astype(np.float32)
    lb = rng.uniform(-5.0, 20.0, rows).astype(np.float32)
    la[:10] = -np.inf          # only b has keys
    lb[10:20] = -np.inf        # only a has keys
    la[20:25] = -np.inf        # neither
    lb[20:25] = -np.inf
    lb[25:35] = la[25:35]      # equal weights
    la[35:40] = lb[35:40] + np.float32(40.0)  # b's weight underflows to 0
    return a, la, b, lb


@pytest.mark.parametrize("d", [64, 128, 256])
def test_merge_matches_oracle(cuda_device, d):
    H.ensure_built()
    rng = np.random.default_rng(30 + d)
    rows = 1003  # not a whole number of blocks or warps
    a, la, b, lb = _states(rng, rows, d)
    ref_out, ref_lse = oracle.merge_states(a.float().numpy(), la, b.float().numpy(), lb)
    dev = cuda_device
    out, lse = _lib.merge_attn_states(a.to(dev), torch.from_numpy(la).to(dev), b.to(dev),
                                      torch.from_numpy(lb).to(dev))
    o = out.float().cpu().numpy().astype(np.float64)
    l = lse.cpu().numpy().astype(np.float64)
    # bf16 rounding of an fp32 result (2^-9 relative), plus fp32 arithmetic on
    # terms that may cancel
    scale = np.abs(a.float().numpy()) + np.abs(b.float().numpy())
    assert np.all(np.abs(o - ref_out) <= 2.0 ** -8 * np.abs(ref_out) + 2.0 ** -18 * scale)
    finite = np.isfinite(ref_lse)
    assert np.all(np.abs(l[finite] - ref_lse[finite]) <= 1e-5 * np.maximum(1.0, np.abs(ref_lse[finite])))
    assert np.all(l[~finite] == -np.inf)
    # exact special cases: an empty side contributes nothing, neither side -> 0
    assert torch.equal(out[:10].cpu(), b[:10])
    assert torch.equal(out[10:20].cpu(), a[10:20])
    assert torch.all(out[20:25].cpu().float() == 0.0)
    assert np.array_equal(l[:10], lb[:10].astype(np.float64))
    assert np.array_equal(l[10:20], la[10:20].astype(np.float64))


def test_merge_in_place_and_without_lse(cuda_device):
    H.ensure_built()
    rng = np.random.default_rng(40)
    rows, d = 777, 128
    a, la, b, lb = _states(rng, rows, d)
    dev = cuda_device
    ref_out, ref_lse = _lib.merge_attn_states(a.to(dev), torch.from_numpy(la).to(dev), b.to(dev),
                                              torch.from_numpy(lb).to(dev))
    # out over out_a, lse over lse_b
    a_dev, la_dev = a.to(dev), torch.from_numpy(la).to(dev)
    b_dev, lb_dev = b.to(dev), torch.from_numpy(lb).to(dev)
    _lib.merge_attn_states(a_dev, la_dev, b_dev, lb_dev, out=a_dev, lse=lb_dev)
    assert torch.equal(a_dev, ref_out)
    assert torch.equal(lb_dev, ref_lse)
    out = _lib.merge_attn_states(a.to(dev), torch.from_numpy(la).to(dev), b.to(dev),
                                 torch.from_numpy(lb).to(dev), return_lse=False)
    assert torch.equal(out, ref_out)
    # [T, Hq, D] shapes, as paged_attention returns them
    out3, lse3 = _lib.merge_attn_states(a.to(dev).reshape(111, 7, d),
                                        torch.from_numpy(la).to(dev).reshape(111, 7),
                                        b.to(dev).reshape(111, 7, d),
                                        torch.from_numpy(lb).to(dev).reshape(111, 7))
    assert torch.equal(out3.reshape(rows, d), ref_out)
    assert torch.equal(lse3.reshape(rows), ref_lse)


@pytest.mark.parametrize("bs,d,splits", [(16, 128, 0), (32, 64, 1), (16, 256, 4)])
def test_two_pass_decode_merged_equals_one_pass(cuda_device, bs, d, splits):
    spec = inputs.Spec(f"merge_decode_{bs}_{d}", 120 + d + bs, hq=16, hk=4, d=d, bs=bs,
                       fixed_decode_lens=(40, 257, 1000, 2049, 64), k_bias_std=SQRT2)
    w = inputs.make_workload(spec)
    g = H.GpuState(w, cuda_device)
    o = H.OracleState(w)
    rows = H.owned_rows(w)
    ref_out, ref_lse = o.attention(rows=rows)
    lens = w.seq_lens.numpy()
    bt = w.block_table.numpy()
    # first part: the first P keys (whole pages); second part: the rest,
    # through the block table shifted by P / bs pages
    p = np.maximum(bs, (lens // 2) // bs * bs).astype(np.int32)
    p = np.minimum(p, lens - 1)
    assert np.all(p % bs == 0) and np.all(p > 0)
    bt2 = np.full_like(bt, -1)
    for s, ps in enumerate(p):
        shifted = bt[s, ps // bs:]
        bt2[s, :shifted.shape[0]] = shifted
    dev = cuda_device
    lens_a = torch.from_numpy(p).to(dev)
    lens_b = torch.from_numpy((lens - p).astype(np.int32)).to(dev)
    bt_b = torch.from_numpy(np.ascontiguousarray(bt2)).to(dev)
    kw = dict(num_splits=splits)
    out_a, lse_a = _lib.paged_attention(g.q, g.kc, g.ks, g.vc, g.vs, g.cu, lens_a,
                                        g.block_table, 1, int(p.max()), w.softmax_scale, **kw)
    out_b, lse_b = _lib.paged_attention(g.q, g.kc, g.ks, g.vc, g.vs, g.cu, lens_b, bt_b, 1,
                                        int((lens - p).max()), w.softmax_scale, **kw)
    out, lse = _lib.merge_attn_states(out_a, lse_a, out_b, lse_b)
    H.compare(out, lse, ref_out, ref_lse, rows, label=f"two-pass merge bs={bs} d={d}")
    full_out, full_lse = g.attention(num_splits=splits)
    diff = (out.float() - full_out.float()).abs().max().item()
    assert diff <= 2e-2, diff
    ldiff = ((lse - full_lse).abs() / full_lse.abs().clamp(min=1.0)).max().item()
    assert ldiff <= 1e-4, ldiff

"""GPU parity at the five serving workloads' full sizes, in the launch
configuration the benchmark times (same seeded inputs, same split count).

The whole q8 cache (codes, scales, placement) is compared bit for bit with
the oracle's own kv_store of the same rows.  Attention is compared element by
element on a sample of (token, q head) rows that the oracle computes one by
one -- random rows plus every sequence's first and last token -- and every
other row is checked against properties that hold at any size: finite values,
and |out| no larger than the largest dequantized |v| (each output is a convex
combination of V rows)."""
import numpy as np
import pytest
import torch

from paged_attention_int8_gb300 import _lib, inputs
from tests import _harness as H

pytestmark = pytest.mark.gpu

FULL = ["decode_batch", "chunked_prefill", "mixed_batch", "long_decode", "long_decode_d256"]


def _edge_rows(w: inputs.Workload) -> np.ndarray:
    """First and last token of every sequence, first and last q head."""
    cu = w.cu_seqlens_q.numpy()
    hq = w.spec.hq
    rows = []
    for s in range(w.num_seqs):
        for tok in {int(cu[s]), int(cu[s + 1]) - 1}:
            rows += [tok * hq, tok * hq + hq - 1]
    return np.asarray(rows, np.int64)


def _max_abs_v(o: H.OracleState) -> float:
    """Largest |code * scale| in the oracle's V cache."""
    scale = o.vs.view(np.float16).astype(np.float32)  # [nb, Hk, G, bs]
    codes = np.abs(o.vc.astype(np.int32)).max()       # |code| <= 127
    return float(codes) * float(np.nanmax(np.abs(scale)))


@pytest.mark.parametrize("name", FULL)
def test_full_size_parity(name, cuda_device):
    spec = inputs.WORKLOADS[name]
    w = inputs.make_workload(spec)
    g = H.GpuState(w, cuda_device)
    o = H.OracleState(w)
    H.assert_cache_equal(g, o)

    # the benchmark's split count: the workload's own, else the library's choice
    ns = spec.num_splits or _lib.auto_num_splits(w.num_seqs, spec.hk, w.max_query_len,
                                                 w.max_seq_len)
    out, lse = g.attention(num_splits=ns)

    rows = np.unique(np.concatenate([H.sample_rows(w, 160, seed=7), _edge_rows(w)]))
    ref_out, ref_lse = o.attention(rows=rows)
    H.compare(out, lse, ref_out, ref_lse, rows, label=f"{name} splits={ns}")

    owned = H.owned_rows(w)
    flat = out.float().reshape(-1, spec.d)[torch.as_tensor(owned, device=out.device)]
    assert bool(torch.isfinite(flat).all()), f"{name}: non-finite output"
    vmax = _max_abs_v(o)
    worst = float(flat.abs().max())
    # bf16 output rounding can lift |out| by one part in 2^8
    assert worst <= vmax * (1 + 2 ** -8), f"{name}: |out| {worst} > max |v| {vmax}"
    lse_all = lse.reshape(-1)[torch.as_tensor(owned, device=lse.device)]
    assert bool(torch.isfinite(lse_all).all()), f"{name}: non-finite lse"

"""The allocation-free entry point, pa_paged_attention_noalloc.

It serves callers that cannot call cudaMalloc (a plugin inside another
framework's executor that forbids allocation, a serving loop that must never
wait on the allocator): the split-KV scratch lives in a static device array
inside the library instead of a caller workspace.  This test calls it through
the C ABI twice in a row -- the second call finds the first call's leftovers
in the shared array -- and checks both results against the regular entry
point, which uses a freshly allocated workspace, and against the CPU oracle,
with the parity tolerances of the other GPU tests.  It lives in a file of its
own, collected last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from paged_attention_int8_gb300 import _lib, inputs
from tests import _harness as H

pytestmark = pytest.mark.gpu

SPEC = inputs.Spec("noalloc_decode", 201, hq=32, hk=8, d=128, bs=16, n_decode=12,
                   decode_lens=(300, 2600), k_bias_std=math.sqrt(2.0))


def _noalloc(lib):
    fn = lib.pa_paged_attention_noalloc
    P, i32 = ctypes.c_void_p, ctypes.c_int32
    fn.argtypes = [P, P, P, P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                   ctypes.c_float, i32, P, P, P, P]
    fn.restype = ctypes.c_int
    return fn


def _call(fn, g, w, num_splits, out, lse, status):
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    s = w.spec
    return fn(p(g.q), p(g.kc), p(g.ks), p(g.vc), p(g.vs), p(g.cu), p(g.seq_lens),
              p(g.block_table), g.block_table.stride(0), w.num_seqs, w.num_tokens, s.hq, s.hk,
              s.d, w.num_blocks, s.bs, w.max_query_len, w.max_seq_len,
              ctypes.c_float(w.softmax_scale), num_splits, p(out), p(lse), p(status),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("num_splits", [0, 16, 1])
def test_noalloc_matches_workspace_entry_on_two_calls(num_splits, cuda_device):
    w = inputs.make_workload(SPEC)
    g = H.GpuState(w, cuda_device)
    lib = _lib.load()
    fn = _noalloc(lib)
    ref_out, ref_lse = g.attention(num_splits=num_splits)
    rows = H.owned_rows(w)
    ref_rows_out = ref_out.float().cpu().numpy().reshape(-1, w.spec.d)[rows].astype(np.float64)
    ref_rows_lse = ref_lse.cpu().numpy().reshape(-1)[rows].astype(np.float64)
    oracle_out, oracle_lse = H.OracleState(w).attention(rows=rows)
    status = torch.full((1,), 7, dtype=torch.int32, device=cuda_device)
    for _ in range(2):
        out = torch.full_like(g.q, float("nan"))
        lse = torch.full((w.num_tokens, w.spec.hq), float("nan"), device=cuda_device)
        st = _call(fn, g, w, num_splits, out, lse, status)
        assert st == _lib.Status.OK, lib.pa_last_error().decode()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        H.compare(out, lse, ref_rows_out, ref_rows_lse, rows, label=f"noalloc splits={num_splits}")
        H.compare(out, lse, oracle_out, oracle_lse, rows,
                  label=f"noalloc vs oracle splits={num_splits}")


def test_noalloc_rejects_splits_beyond_its_scratch(cuda_device):
    # 2048 single-token sequences x 32 heads x 16 splits x 130 floats > 8 MiB
    lib = _lib.load()
    fn = _noalloc(lib)
    dummy = torch.zeros(64, dtype=torch.uint8, device=cuda_device)
    p = ctypes.c_void_p(dummy.data_ptr())
    st = fn(p, p, p, p, p, p, p, p, 4, 2048, 2048, 32, 8, 128, 16, 16, 1, 8192,
            ctypes.c_float(0.1), 16, p, p, None, None)
    assert st == _lib.Status.INVALID_ARG
    assert "static scratch" in lib.pa_last_error().decode()


def test_noalloc_binding_matches_the_raw_call(cuda_device):
    # the thin binding marshals the same arguments as the raw C call
    w = inputs.make_workload(SPEC)
    g = H.GpuState(w, cuda_device)
    lib = _lib.load()
    fn = _noalloc(lib)
    status = torch.zeros(1, dtype=torch.int32, device=cuda_device)
    raw_out = torch.full_like(g.q, float("nan"))
    raw_lse = torch.full((w.num_tokens, w.spec.hq), float("nan"), device=cuda_device)
    assert _call(fn, g, w, 0, raw_out, raw_lse, status) == _lib.Status.OK
    out, lse = _lib.paged_attention_noalloc(g.q, g.kc, g.ks, g.vc, g.vs, g.cu, g.seq_lens,
                                            g.block_table, w.max_query_len, w.max_seq_len,
                                            w.softmax_scale, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(out, raw_out)
    assert torch.equal(lse, raw_lse)

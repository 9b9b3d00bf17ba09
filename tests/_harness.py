"""Shared set-up for the GPU parity tests: the same seeded workload goes
through the CUDA library (via the C ABI binding) and through the CPU oracle,
and the results are compared.  The oracle only ever sees the generated host
inputs, never anything the GPU produced."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from paged_attention_int8_gb300 import _lib, build as pkg_build, inputs

# Tolerances of the method statement: bit-exact q8 cache; output max|err| <= 1e-2
# and mean|err| <= 1e-3 against the fp64 oracle; LSE |err| <= 1e-4 * max(1, |lse|).
OUT_MAX = 1e-2
OUT_MEAN = 1e-3
LSE_REL = 1e-4

_built = False


def ensure_built():
    global _built
    if not _built:
        pkg_build.build()
        _built = True


class GpuState:
    """Device tensors of a workload; the cache filled by the library's kv_store."""

    def __init__(self, w: inputs.Workload, device, populate: bool = True):
        ensure_built()
        s = w.spec
        self.w = w
        self.device = device
        self.kc, self.ks, self.vc, self.vs = inputs.empty_cache(w.num_blocks, s.hk, s.bs, s.d,
                                                                device=device)
        self.status = torch.zeros(4, dtype=torch.int32, device=device)
        self.q = w.q.to(device)
        self.cu = w.cu_seqlens_q.to(device)
        self.seq_lens = w.seq_lens.to(device)
        self.block_table = w.block_table.to(device)
        if populate:
            self.store(w.prefix_key, w.prefix_value, w.prefix_slots)
            self.store(w.new_key, w.new_value, w.new_slots)

    def store(self, key, value, slots):
        if key.shape[0] == 0:
            return
        _lib.kv_store(key.to(self.device), value.to(self.device), slots.to(self.device),
                      self.kc, self.ks, self.vc, self.vs, status=self.status)
        assert _lib.check_status(self.status) == 0

    def attention(self, num_splits=None, max_query_len=None, max_seq_len=None, lse=True):
        w = self.w
        ns = w.spec.num_splits if num_splits is None else num_splits
        need = _lib.workspace_size(w.num_seqs, w.spec.hq, w.spec.d, ns)
        ws = torch.zeros(need, dtype=torch.uint8, device=self.device)
        out = torch.full_like(self.q, float("nan"))
        lse_t = torch.full((w.num_tokens, w.spec.hq), float("nan"), device=self.device) if lse else None
        _lib.paged_attention(self.q, self.kc, self.ks, self.vc, self.vs, self.cu, self.seq_lens,
                             self.block_table, max_query_len or w.max_query_len,
                             max_seq_len or w.max_seq_len, w.softmax_scale, num_splits=ns,
                             out=out, lse=lse_t, workspace=ws, return_lse=lse)
        bits = _lib.check_status(ws)
        assert bits == 0
        return out, lse_t


class OracleState:
    """Host caches written by the oracle's own kv_store from the generated rows."""

    def __init__(self, w: inputs.Workload):
        s = w.spec
        self.w = w
        kc, ks, vc, vs = inputs.empty_cache(w.num_blocks, s.hk, s.bs, s.d)
        self.kc, self.vc = kc.numpy(), vc.numpy()
        self.ks, self.vs = ks.numpy().view(np.uint16), vs.numpy().view(np.uint16)
        for k, v, sl in ((w.prefix_key, w.prefix_value, w.prefix_slots),
                         (w.new_key, w.new_value, w.new_slots)):
            if k.shape[0]:
                bad = oracle.kv_store(inputs.bf16_bits(k), inputs.bf16_bits(v), sl.numpy(),
                                      self.kc, self.ks, self.vc, self.vs)
                assert bad == 0

    def attention(self, rows=None):
        w = self.w
        return oracle.paged_attention(inputs.bf16_bits(w.q), self.kc, self.ks, self.vc, self.vs,
                                      w.cu_seqlens_q.numpy(), w.seq_lens.numpy(),
                                      w.block_table.numpy(), w.softmax_scale, rows=rows)


def assert_cache_equal(g: GpuState, o: OracleState):
    np.testing.assert_array_equal(g.kc.cpu().numpy(), o.kc)
    np.testing.assert_array_equal(g.vc.cpu().numpy(), o.vc)
    np.testing.assert_array_equal(g.ks.cpu().numpy().view(np.uint16), o.ks)
    np.testing.assert_array_equal(g.vs.cpu().numpy().view(np.uint16), o.vs)


def owned_rows(w: inputs.Workload) -> np.ndarray:
    """Row ids (token * Hq + head) of tokens some sequence owns."""
    cu = w.cu_seqlens_q.numpy()
    toks = np.concatenate([np.arange(cu[s], cu[s + 1]) for s in range(w.num_seqs)] or [[]])
    toks = toks.astype(np.int64)
    hq = w.spec.hq
    return (toks[:, None] * hq + np.arange(hq)[None, :]).reshape(-1)


def compare(out_gpu: torch.Tensor, lse_gpu, out_ref: np.ndarray, lse_ref: np.ndarray,
            rows: np.ndarray, label: str = ""):
    """Element-wise comparison of GPU rows with oracle rows (same order)."""
    hq = out_gpu.shape[1]
    d = out_gpu.shape[2]
    o = out_gpu.float().cpu().numpy().reshape(-1, d)[rows].astype(np.float64)
    err = np.abs(o - out_ref)
    assert np.all(np.isfinite(o)), f"{label}: non-finite output"
    max_err, mean_err = float(err.max()), float(err.mean())
    assert max_err <= OUT_MAX, f"{label}: output max|err| {max_err:.3e} > {OUT_MAX}"
    assert mean_err <= OUT_MEAN, f"{label}: output mean|err| {mean_err:.3e} > {OUT_MEAN}"
    stats = dict(out_max=max_err, out_mean=mean_err)
    if lse_gpu is not None:
        lg = lse_gpu.cpu().numpy().reshape(-1)[rows].astype(np.float64)
        lerr = np.abs(lg - lse_ref) / np.maximum(1.0, np.abs(lse_ref))
        assert np.all(np.isfinite(lg)), f"{label}: non-finite lse"
        worst = float(lerr.max())
        assert worst <= LSE_REL, f"{label}: lse rel err {worst:.3e} > {LSE_REL}"
        stats["lse_rel_max"] = worst
    return stats


def check_workload(w: inputs.Workload, device, splits=(None,), rows=None, cache=True, **kw):
    g = GpuState(w, device)
    o = OracleState(w)
    if cache:
        assert_cache_equal(g, o)
    all_rows = owned_rows(w)
    rows = all_rows if rows is None else np.asarray(rows, np.int64)
    ref_out, ref_lse = o.attention(rows=rows)
    results = {}
    for ns in splits:
        out, lse = g.attention(num_splits=ns, **kw)
        results[ns] = compare(out, lse, ref_out, ref_lse, rows, label=f"{w.spec.name} splits={ns}")
        # rows no sequence owns stay untouched
        owned = np.zeros(w.num_tokens * w.spec.hq, bool)
        owned[all_rows] = True
        flat = out.float().cpu().numpy().reshape(-1, w.spec.d)
        assert np.all(np.isnan(flat[~owned]))
    return g, o, results


def sample_rows(w: inputs.Workload, n: int, seed: int = 0) -> np.ndarray:
    rows = owned_rows(w)
    rng = np.random.default_rng(seed)
    pick = rng.choice(rows.shape[0], size=min(n, rows.shape[0]), replace=False)
    # always include each sequence's last token's first head and the first token
    return np.unique(np.concatenate([rows[pick], rows[:1], rows[-1:]]))


def rel_lse_tol(lse):
    return LSE_REL * max(1.0, abs(lse))


__all__ = ["GpuState", "OracleState", "assert_cache_equal", "compare", "check_workload",
           "owned_rows", "sample_rows", "ensure_built", "math"]

"""Host-side arithmetic of bench.py, checked on the CPU: the algorithmic
work of a step (visible (row, key) pairs, KV and store bytes) against
brute-force counts, and the rule that a recorded ncu traffic figure holds
only while the attention kernels' sources are unchanged."""
import os
import shutil

import numpy as np
import pytest

import bench
from paged_attention_int8_gb300 import inputs

SPECS = [
    inputs.TINY_DECODE,
    inputs.Spec("cpu_prefill", 201, hq=8, hk=2, d=64, bs=16, n_prefill=3, prefill_qlen=37,
                prefix_lens=(0, 90)),
    inputs.Spec("cpu_mixed", 202, hq=8, hk=4, d=128, bs=32, n_prefill=2, prefill_qlen=20,
                prefix_lens=(5, 40), n_decode=4, decode_lens=(1, 130), pad_frac=0.1),
]


@pytest.mark.parametrize("spec", SPECS, ids=lambda s: s.name)
def test_step_work_matches_brute_force_counts(spec):
    w = inputs.make_workload(spec)
    cu = w.cu_seqlens_q.numpy()
    lens = w.seq_lens.numpy()
    pairs = 0
    keys = 0
    pages = 0
    for s in range(w.num_seqs):
        q_len = int(cu[s + 1] - cu[s])
        ctx = int(lens[s]) - q_len
        for i in range(q_len):          # query i of the chunk sees keys 0 .. ctx + i
            pairs += sum(1 for j in range(int(lens[s])) if j <= ctx + i)
        keys += int(lens[s])
        pages += -(-int(lens[s]) // spec.bs)
    g = spec.d // 32
    work = bench.step_work(w)
    assert work["pairs"] == pairs * spec.hq
    assert work["flops"] == 4 * spec.d * pairs * spec.hq
    assert work["kv_bytes"] == keys * spec.hk * 2 * (spec.d + 2 * g)
    t = w.num_tokens
    assert work["attn_bytes"] == (work["kv_bytes"] + t * spec.hq * spec.d * 4 + t * spec.hq * 4
                                  + 4 * pages + 4 * (2 * w.num_seqs + 1))
    slots = w.new_slots.numpy()
    stored = int(np.sum(slots >= 0))
    assert stored < slots.shape[0] or spec.pad_frac == 0.0
    assert work["store_bytes"] == (stored * spec.hk * (4 * spec.d + 2 * (spec.d + 2 * g))
                                   + 8 * slots.shape[0])
    assert work["step_bytes"] == work["attn_bytes"] + work["store_bytes"]


def test_recorded_traffic_holds_only_for_the_same_attention_sources(tmp_path, monkeypatch):
    csrc = os.path.join(bench.ROOT, "paged_attention_int8_gb300", "csrc")
    shutil.copytree(csrc, tmp_path / "paged_attention_int8_gb300" / "csrc")
    (tmp_path / "profiles").mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    sha = bench.kernel_sources_sha256()
    (tmp_path / "profiles" / "attention_x.md").write_text(
        f"# x\n\ntraffic_bytes_per_launch: 123456\nsource_sha256: {sha}\n")
    assert bench.recorded_traffic("x") == 123456.0
    assert bench.recorded_traffic("missing") is None
    # a change outside the attention kernels keeps the figure
    other = tmp_path / "paged_attention_int8_gb300" / "csrc" / "kv_store.cu"
    other.write_text(other.read_text() + "\n// edit\n")
    assert bench.recorded_traffic("x") == 123456.0
    # a change to a source of the attention kernels drops it
    attn = tmp_path / "paged_attention_int8_gb300" / "csrc" / "attn_decode.cu"
    attn.write_text(attn.read_text() + "\n// edit\n")
    assert bench.recorded_traffic("x") is None


def test_roofline_reports_both_parts_for_a_mixed_batch():
    spec = SPECS[2]
    w = inputs.make_workload(spec)
    work = bench.step_work(w)
    roof = bench.roofline_of("cpu_mixed", spec, w, work, attn_ms=0.5, ns_eff=2,
                             hbm_peak=6000.0, tc_peak=2000.0, peak_src="test")
    parts = roof["parts"]
    assert roof["bound"] == "hbm" and roof["unit"] == "GB/s"
    assert parts["bytes_ms"] == pytest.approx(work["attn_bytes"] / 6000e9 * 1e3, abs=2e-6)
    assert parts["flops_ms"] == pytest.approx(work["flops"] / 2000e12 * 1e3, abs=2e-6)
    assert parts["roofline_ms"] == max(parts["bytes_ms"], parts["flops_ms"])
    assert roof["frac"] == pytest.approx(work["attn_bytes"] / 0.5e-3 / 6000e9, abs=1e-4)
    prefill = bench.roofline_of("cpu_prefill", SPECS[1], inputs.make_workload(SPECS[1]),
                                bench.step_work(inputs.make_workload(SPECS[1])), attn_ms=1.0,
                                ns_eff=1, hbm_peak=6000.0, tc_peak=2000.0, peak_src="test")
    assert prefill["bound"] == "tensor" and "parts" not in prefill


def test_the_suite_holds_every_serving_workload_and_the_headline_is_the_largest():
    assert set(bench.SUITE) == set(inputs.WORKLOADS) - {"tiny_decode"}
    kv = {n: bench.step_work(inputs.make_workload(inputs.WORKLOADS[n].replace(
        fixed_decode_lens=tuple(min(L, 4096) for L in inputs.WORKLOADS[n].fixed_decode_lens))))
        ["kv_bytes"] for n in ("long_decode", "long_decode_d256")}
    assert kv["long_decode_d256"] > kv["long_decode"]
    assert bench.HEADLINE == "long_decode_d256"

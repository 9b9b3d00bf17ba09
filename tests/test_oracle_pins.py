"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests re-types the oracle's formulas.  Each one checks the
oracle against something else: values worked out by hand from the pages'
definitions (tests/golden), a library routine (numpy's IEEE fp16 conversion,
torch's fp64 scaled_dot_product_attention and logsumexp), closed forms,
invariants, or one part of the oracle against another (split against joint).
"""
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_attention_int8_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "q8_hand_examples.txt")


# ----------------------------------------------------------------------------- helpers

def _load_golden():
    cases = []
    for line in open(GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, xs, codes, bits = [p.strip() for p in line.split(";")]
        x = np.array([float(v) for v in xs.split(",")], np.float32)
        c = np.array([int(v) for v in codes.split(",")], np.int8)
        cases.append((name, x, c, int(bits, 16)))
    return cases


def _f16_bits_numpy(x: np.ndarray) -> np.ndarray:
    return np.asarray(x, np.float32).astype(np.float16).view(np.uint16)


def _bf16_bits(x: torch.Tensor) -> np.ndarray:
    return inputs.bf16_bits(x.to(torch.bfloat16))


def _rand_cache(rng, num_blocks, hk, bs, d, scale_lo=0.005, scale_hi=0.05):
    kcs, kss, vcs, vss = inputs.cache_shapes(num_blocks, hk, bs, d)
    kc = rng.integers(-127, 128, size=kcs, dtype=np.int8)
    vc = rng.integers(-127, 128, size=vcs, dtype=np.int8)
    ks = _f16_bits_numpy(rng.uniform(scale_lo, scale_hi, size=kss))
    vs = _f16_bits_numpy(rng.uniform(scale_lo, scale_hi, size=vss))
    return kc, ks, vc, vs


def _dequant(codes, scales):
    """Reference dequantization with numpy (fp64): value = code * fp16 scale,
    token-major pages [..., bs, D] with scales [..., bs, D/32]."""
    s = scales.view(np.float16).astype(np.float64)
    return codes.astype(np.float64) * np.repeat(s, 32, axis=-1)


def _token_major_v(vc, vs):
    """Channel-major V pages [nb, hk, D, bs] / [nb, hk, D/32, bs] viewed
    token-major, for the numpy references."""
    return (np.ascontiguousarray(vc.transpose(0, 1, 3, 2)),
            np.ascontiguousarray(vs.transpose(0, 1, 3, 2)))


def _problem(rng, q_lens, seq_lens, hq, hk, d, bs, spare=3, q_scale=1.0):
    S = len(seq_lens)
    pages = [(L + bs - 1) // bs for L in seq_lens]
    num_blocks = sum(pages) + spare
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((S, max(pages)), -1, np.int32)
    pos = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    cu = np.zeros(S + 1, np.int32)
    cu[1:] = np.cumsum(q_lens)
    T = int(cu[-1])
    q = _bf16_bits(torch.from_numpy(rng.standard_normal((T, hq, d)) * q_scale))
    kc, ks, vc, vs = _rand_cache(rng, num_blocks, hk, bs, d)
    return dict(q=q, kc=kc, ks=ks, vc=vc, vs=vs, cu=cu, sl=np.array(seq_lens, np.int32),
                bt=bt, hq=hq, hk=hk, d=d, bs=bs)


def _run(p, scale, rows=None):
    return oracle.paged_attention(p["q"], p["kc"], p["ks"], p["vc"], p["vs"], p["cu"],
                                  p["sl"], p["bt"], scale, rows=rows, n_threads=4)


def _gather(p, codes, scales, s, L):
    """Logical [L, Hk, D] fp64 of sequence s (numpy gather through the table).
    V pages (channel-major) are recognised by their shape and transposed."""
    bs = p["bs"]
    if codes.shape[2] != bs:  # V: [nb, hk, D, bs] (D >= 64 > bs)
        codes, scales = _token_major_v(codes, scales)
    j = np.arange(L)
    blk = p["bt"][s, j // bs]
    off = j % bs
    deq = _dequant(codes, scales)                 # [nb, hk, bs, d]
    return deq[blk, :, off, :]                     # [L, hk, d]


# ----------------------------------------------------------------------------- number formats

def test_f16_conversion_matches_ieee_round_to_nearest_even():
    rng = np.random.default_rng(11)
    vals = [rng.standard_normal(4000) * 10.0 ** rng.integers(-9, 5, 4000)]
    # exact midpoints between neighbouring fp16 values (ties), normal and subnormal
    h = np.arange(0, 0x7bff, 7, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    vals.append(((lo + hi) / 2).astype(np.float32))
    vals.append(np.array([0.0, -0.0, 1e-8, 2.98e-8, 2.9802322e-08, 5.96e-8, 6.1e-5,
                          65504.0, 65519.99, 65520.0, 65536.0, 1e30, -65520.0,
                          np.float32(1) / np.float32(127)], np.float32))
    x = np.concatenate([np.asarray(v, np.float32) for v in vals])
    x = np.concatenate([x, -x])
    got = np.array([oracle.f32_to_f16_bits(float(v)) for v in x], np.uint16)
    np.testing.assert_array_equal(got, _f16_bits_numpy(x))


def test_f16_decode_matches_ieee_for_every_finite_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = np.isfinite(bits.view(np.float16))
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_bits_to_f32(int(b)) for b in bits[finite]], np.float32)
    np.testing.assert_array_equal(got, ref[finite])


# ----------------------------------------------------------------------------- q8 quantizer

@pytest.mark.parametrize("case", _load_golden(), ids=lambda c: c[0])
def test_q8_hand_examples(case):
    name, x, codes, bits = case
    got_codes, got_bits = oracle.q8_quantize_group(x)
    np.testing.assert_array_equal(got_codes, codes)
    assert got_bits == bits


def test_q8_rounding_is_half_away_not_half_even_nor_add_half_truncate():
    # 0.5 - 2^-25: exact rounding gives 0; "+0.5 then truncate" in fp32 gives 1
    # (0.5 - 2^-25 + 0.5 rounds up to 1.0), and half-even would also give 0.
    x = np.zeros(32, np.float32)
    x[0] = 127.0
    x[1] = np.float32(0.5) - np.float32(2.0 ** -25)
    x[2] = 2.5
    codes, _ = oracle.q8_quantize_group(x)
    assert codes[1] == 0
    assert codes[2] == 3  # half-even would give 2


def _random_groups(rng, n):
    groups = []
    for i in range(n):
        kind = i % 5
        if kind == 0:
            g = rng.standard_normal(32)
        elif kind == 1:   # one outlier over tiny values
            g = rng.standard_normal(32) * 1e-3
            g[rng.integers(32)] = rng.choice([-1, 1]) * rng.uniform(10, 1000)
        elif kind == 2:   # values on tie points of a scale-one grid
            g = rng.integers(-126, 127, 32) + 0.5
            g[0] = 127.0
        elif kind == 3:   # widely varying magnitudes
            g = rng.standard_normal(32) * 10.0 ** rng.uniform(-6, 4)
        else:             # bf16-representable values, as the kernels see them
            g = torch.from_numpy(rng.standard_normal(32) * 3).to(torch.bfloat16).float().numpy()
        groups.append(np.asarray(g, np.float32))
    return groups


def test_q8_invariants_on_random_groups():
    rng = np.random.default_rng(5)
    for x in _random_groups(rng, 600):
        codes, bits = oracle.q8_quantize_group(x)
        c = codes.astype(np.int64)
        amax = float(np.max(np.abs(x)))
        s16 = float(np.array([bits], np.uint16).view(np.float16)[0])
        assert np.all(np.abs(c) <= 127)
        assert not np.any(c == -128)
        # the element of largest magnitude maps to +-127
        k = int(np.argmax(np.abs(x)))
        if amax > 0:
            assert c[k] == (127 if x[k] > 0 else -127)
        # rounding error against the fp32 scale: at most half a step (plus the
        # quotient's own rounding), never more
        s32 = max(amax / 127.0, 1e-8)
        err = np.abs(x.astype(np.float64) - c * s32)
        assert np.all(err <= 0.5 * s32 * (1 + 1e-6) + 1e-30)
        # round trip through the stored fp16 scale
        rt = np.abs(x.astype(np.float64) - c * s16)
        assert np.all(rt <= 0.5 * s32 * (1 + 1e-6) + 127 * abs(s32 - s16) + 1e-30)
        # the fp16 scale is the nearest fp16 of the fp32 scale: within half an ulp
        assert abs(s16 - s32) <= 2.0 ** -11 * s32 + 2.0 ** -25


def test_q8_groups_are_32_consecutive_channels():
    # Four groups with very different magnitudes: each group's scale depends on
    # its own 32 channels only, so each group's maximum maps to 127.
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(32) * m for m in (1e-3, 1.0, 50.0, 1e-6)])
    bits = _bf16_bits(torch.from_numpy(x)).reshape(1, 128)
    codes, scales = oracle.q8_quantize_rows(bits)
    xb = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()[0]
    for g in range(4):
        part = xb[32 * g:32 * g + 32]
        one_codes, one_bits = oracle.q8_quantize_group(part)
        np.testing.assert_array_equal(codes[0, 32 * g:32 * g + 32], one_codes)
        assert scales[0, g] == one_bits
        assert np.max(np.abs(codes[0, 32 * g:32 * g + 32].astype(int))) == 127


# ----------------------------------------------------------------------------- kv_store scatter

def _small_store_problem(seed=0, hk=2, d=64, bs=16):
    spec = inputs.Spec("pin", seed, hq=2 * hk, hk=hk, d=d, bs=bs, n_prefill=2, prefill_qlen=5,
                       prefix_lens=(3, 40), n_decode=3, decode_lens=(1, 50), pad_frac=0.2,
                       spare_blocks=4)
    return inputs.make_workload(spec)


def test_kv_store_skips_padding_and_leaves_canary_elsewhere():
    w = _small_store_problem()
    k, v, slots = w.all_key_value()
    kc, ks, vc, vs = [t.numpy() for t in inputs.empty_cache(w.num_blocks, 2, 16, 64)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    bad = oracle.kv_store(inputs.bf16_bits(k), inputs.bf16_bits(v), slots.numpy(), kc, ks, vc, vs)
    assert bad == 0
    written = np.zeros(w.num_blocks * 16, bool)
    written[slots.numpy()[slots.numpy() >= 0]] = True
    # slot -> (block, offset) in HND: a written slot holds no canary, an
    # unwritten one holds only canary
    codes_by_slot = kc.transpose(0, 2, 1, 3).reshape(w.num_blocks * 16, -1)
    scales_by_slot = ks.transpose(0, 2, 1, 3).reshape(w.num_blocks * 16, -1)
    assert np.all(codes_by_slot[~written] == -128)
    assert np.all(scales_by_slot[~written] == 0xFFFF)
    assert not np.any(codes_by_slot[written] == -128)
    assert (slots.numpy() < 0).sum() > 0  # padding rows were present and skipped


def test_kv_store_out_of_range_slot_is_reported_not_written():
    kc, ks, vc, vs = [t.numpy() for t in inputs.empty_cache(2, 1, 16, 32)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    key = _bf16_bits(torch.ones(3, 1, 32))
    bad = oracle.kv_store(key, key, np.array([5, 32, -1], np.int64), kc, ks, vc, vs)
    assert bad == 1
    assert np.all(kc.reshape(32, 32)[np.arange(32) != 5] == -128)


def test_store_then_gather_is_independent_of_physical_placement():
    # The same rows stored under two different block tables read back equal
    # through each table: placement is invisible to a reader of the logical cache.
    w1 = _small_store_problem(seed=1)
    logical = []
    rng = np.random.default_rng(9)
    perm = rng.permutation(w1.num_blocks).astype(np.int32)
    bt2 = np.where(w1.block_table.numpy() >= 0, perm[np.maximum(w1.block_table.numpy(), 0)], -1)
    k, v, slots = w1.all_key_value()
    slots = slots.numpy()
    bs = 16
    slots2 = np.where(slots >= 0, perm[np.maximum(slots, 0) // bs] * bs + np.maximum(slots, 0) % bs, -1)
    for table, sl in ((w1.block_table.numpy(), slots), (bt2, slots2)):
        kc, ks, vc, vs = [t.numpy() for t in inputs.empty_cache(w1.num_blocks, 2, bs, 64)]
        ks, vs = ks.view(np.uint16), vs.view(np.uint16)
        oracle.kv_store(inputs.bf16_bits(k), inputs.bf16_bits(v), sl, kc, ks, vc, vs)
        p = dict(bt=table, bs=bs)
        logical.append([_gather(p, kc, ks, s, int(L)) for s, L in enumerate(w1.seq_lens.tolist())]
                       + [_gather(p, vc, vs, s, int(L)) for s, L in enumerate(w1.seq_lens.tolist())])
    for a, b in zip(*logical):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("d,bs", [(64, 16), (128, 32), (256, 16)])
def test_kv_store_places_each_tokens_quantized_row_at_its_slot(d, bs):
    """What lands where: for every (token, kv head) with a slot, the codes and
    fp16 scale bits read back at (slot // bs, head, slot % bs) -- token-major
    K rows, channel-major V columns, read here with numpy indexing written from
    the page layout -- equal the quantized source row of that token and head
    (block = slot // block_size, offset = slot % block_size, as in
    "attention_impl.py", `_store_kvcache_nhd`), and dequantize to within the
    q8 round-trip bound of the bf16 source ("shared/attention_kit.py",
    `quantize_q8`).  Heads get magnitudes 10^(h-1) and K / V different ones,
    so a head or K/V exchange, or a transposed V page, breaks both checks."""
    hk = 3
    rng = np.random.default_rng(40 + d)
    n_tok = 3 * bs + 5
    num_blocks = n_tok // bs + 4
    # distinct slots in shuffled blocks, ragged offsets, a few padding rows
    slots = rng.permutation(num_blocks * bs)[:n_tok].astype(np.int64)
    slots[rng.choice(n_tok, size=4, replace=False)] = -1
    mag_k = 10.0 ** (np.arange(hk) - 1.0)
    mag_v = 3.0 * 10.0 ** (1.0 - np.arange(hk))
    k = torch.from_numpy(rng.standard_normal((n_tok, hk, d)) * mag_k[None, :, None])
    v = torch.from_numpy(rng.standard_normal((n_tok, hk, d)) * mag_v[None, :, None])
    kb, vb = _bf16_bits(k), _bf16_bits(v)
    kc, ks, vc, vs = [t.numpy() for t in inputs.empty_cache(num_blocks, hk, bs, d)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    assert oracle.kv_store(kb, vb, slots, kc, ks, vc, vs) == 0
    src = {"k": torch.from_numpy(kb.view(np.int16)).view(torch.bfloat16).double().numpy(),
           "v": torch.from_numpy(vb.view(np.int16)).view(torch.bfloat16).double().numpy()}
    checked = 0
    for n in range(n_tok):
        slot = int(slots[n])
        if slot < 0:
            continue
        blk, off = slot // bs, slot % bs
        for h in range(hk):
            got = {"k": (kc[blk, h, off, :], ks[blk, h, off, :]),
                   "v": (vc[blk, h, :, off], vs[blk, h, :, off])}
            for name, bits in (("k", kb), ("v", vb)):
                codes, scales = got[name]
                want_c, want_s = oracle.q8_quantize_rows(bits[n, h][None, :])
                np.testing.assert_array_equal(codes, want_c[0], err_msg=f"{name} n={n} h={h}")
                np.testing.assert_array_equal(scales, want_s[0], err_msg=f"{name} n={n} h={h}")
                s16 = np.repeat(scales.view(np.float16).astype(np.float64), 32)
                x = src[name][n, h]
                # |x - code * s16| <= s32/2 + 127 |s32 - s16| with |s32 - s16| <= 2^-11 s32
                bound = s16 * (0.5 + 127 * 2.0 ** -11) * (1 + 2.0 ** -10)
                assert np.all(np.abs(x - codes.astype(np.float64) * s16) <= bound), (name, n, h)
                # each group's largest magnitude maps to +-127
                assert np.all(np.abs(codes.reshape(-1, 32)).max(axis=1) == 127)
            checked += 1
    assert checked == (n_tok - 4) * hk
    # every unwritten slot still holds the canary, in K and in V
    written = np.zeros(num_blocks * bs, bool)
    written[slots[slots >= 0]] = True
    unw = np.nonzero(~written)[0]
    assert np.all(kc[unw // bs, :, unw % bs, :] == -128)
    assert np.all(vc.transpose(0, 3, 1, 2)[unw // bs, unw % bs] == -128)
    assert np.all(vs.transpose(0, 3, 1, 2)[unw // bs, unw % bs] == 0xFFFF)


# ----------------------------------------------------------------------------- attention

def test_attention_matches_torch_sdpa_fp64_brute_force():
    """Tiny mixed batch against torch's scaled_dot_product_attention in float64
    (explicit causal mask with key offset k_len - q_len, repeat_interleave of
    kv heads), as the torch reference paths of "attention_impl.py" set it up;
    LSE against torch.logsumexp of the masked scores."""
    rng = np.random.default_rng(21)
    hq, hk, d, bs = 6, 2, 64, 16
    q_lens = [5, 1, 3, 1, 17]
    seq_lens = [5, 40, 19, 1, 50]
    p = _problem(rng, q_lens, seq_lens, hq, hk, d, bs)
    scale = 0.125
    out, lse = _run(p, scale)
    out = out.reshape(-1, hq, d)
    lse = lse.reshape(-1, hq)
    qf = torch.from_numpy(p["q"].view(np.int16)).view(torch.bfloat16).double()
    for s in range(len(q_lens)):
        L, ql = seq_lens[s], q_lens[s]
        K = torch.from_numpy(_gather(p, p["kc"], p["ks"], s, L))          # [L, hk, d]
        V = torch.from_numpy(_gather(p, p["vc"], p["vs"], s, L))
        K = K.repeat_interleave(hq // hk, dim=1).transpose(0, 1)          # [hq, L, d]
        V = V.repeat_interleave(hq // hk, dim=1).transpose(0, 1)
        Q = qf[p["cu"][s]:p["cu"][s + 1]].transpose(0, 1)                  # [hq, ql, d]
        mask = torch.arange(L)[None, :] <= (L - ql + torch.arange(ql))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(
            Q[None], K[None], V[None], attn_mask=mask, scale=scale)[0].transpose(0, 1)
        scores = (Q @ K.transpose(1, 2)) * scale
        ref_lse = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1).transpose(0, 1)
        np.testing.assert_allclose(out[p["cu"][s]:p["cu"][s + 1]], ref.numpy(), rtol=0, atol=1e-12)
        np.testing.assert_allclose(lse[p["cu"][s]:p["cu"][s + 1]], ref_lse.numpy(), rtol=0, atol=1e-12)


def _run_opt(p, scale, **kw):
    return oracle.paged_attention(p["q"], p["kc"], p["ks"], p["vc"], p["vs"], p["cu"],
                                  p["sl"], p["bt"], scale, n_threads=4, **kw)


def _sdpa_masked(p, scale, mask_fn):
    """Per-sequence fp64 SDPA with an explicit boolean mask mask_fn(L, ql) ->
    [ql, L], and the logsumexp of the masked scores (rows with no visible key
    give out 0 and -inf here, as the oracle defines them)."""
    hq, hk, d = p["hq"], p["hk"], p["d"]
    qf = torch.from_numpy(p["q"].view(np.int16)).view(torch.bfloat16).double()
    outs, lses = [], []
    for s in range(len(p["sl"])):
        L, ql = int(p["sl"][s]), int(p["cu"][s + 1] - p["cu"][s])
        Q = qf[p["cu"][s]:p["cu"][s + 1]].transpose(0, 1)                  # [hq, ql, d]
        if L == 0:
            outs.append(np.zeros((ql, hq, d)))
            lses.append(np.full((ql, hq), -np.inf))
            continue
        K = torch.from_numpy(_gather(p, p["kc"], p["ks"], s, L))
        V = torch.from_numpy(_gather(p, p["vc"], p["vs"], s, L))
        K = K.repeat_interleave(hq // hk, dim=1).transpose(0, 1)
        V = V.repeat_interleave(hq // hk, dim=1).transpose(0, 1)
        mask = mask_fn(L, ql)
        scores = ((Q @ K.transpose(1, 2)) * scale).masked_fill(~mask, float("-inf"))
        lse = torch.logsumexp(scores, dim=-1)
        out = torch.softmax(scores, dim=-1) @ V
        outs.append(out.transpose(0, 1).numpy())
        lses.append(lse.transpose(0, 1).numpy())
    return np.concatenate(outs).reshape(-1, d), np.concatenate(lses).reshape(-1)


@pytest.mark.parametrize("window", [1, 3, 16, 37])
def test_sliding_window_matches_torch_brute_force(window):
    # "attention_impl.py": window_size = (sliding_window - 1, 0) -- the query
    # at absolute position p sees keys p - (W - 1) .. p
    rng = np.random.default_rng(31)
    p = _problem(rng, [4, 1, 9, 2], [60, 33, 9, 70], 6, 2, 64, 16)
    scale = 0.125
    out, lse = _run_opt(p, scale, window=window)

    def band(L, ql):
        pos = L - ql + torch.arange(ql)[:, None]
        j = torch.arange(L)[None, :]
        return (j <= pos) & (j >= pos - (window - 1))
    ref, ref_lse = _sdpa_masked(p, scale, band)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_sliding_window_special_cases():
    rng = np.random.default_rng(32)
    p = _problem(rng, [3, 1], [40, 25], 4, 2, 64, 16)
    scale = 0.2
    full = _run(p, scale)
    wide = _run_opt(p, scale, window=40)            # covers every visible key
    np.testing.assert_array_equal(wide[0], full[0])
    np.testing.assert_array_equal(wide[1], full[1])
    one = _run_opt(p, scale, window=1)              # only the query's own position
    qf = torch.from_numpy(p["q"].view(np.int16)).view(torch.bfloat16).double().numpy()
    for s, (t0, t1) in enumerate(((0, 3), (3, 4))):
        L = int(p["sl"][s])
        K = _gather(p, p["kc"], p["ks"], s, L)
        V = _gather(p, p["vc"], p["vs"], s, L)
        for t in range(t0, t1):
            pos = L - (t1 - t0) + (t - t0)
            for h in range(4):
                r = t * 4 + h
                np.testing.assert_allclose(one[0][r], V[pos, h // 2], rtol=0, atol=1e-15)
                sc = np.float64(np.float32(scale)) * float(qf[t, h] @ K[pos, h // 2])
                assert abs(one[1][r] - sc) < 1e-12


def test_sinks_closed_form():
    # "triton_turboquant_unified_attention.py", USE_SINKS: out = sum_i
    # exp(s_i) v_i / (exp(sink) + sum_i exp(s_i)); so out_sink = out *
    # sigmoid(lse - sink) and lse_sink = logaddexp(lse, sink)
    rng = np.random.default_rng(33)
    p = _problem(rng, [5, 1, 2], [50, 17, 2], 6, 3, 64, 16)
    scale = 0.125
    out, lse = _run(p, scale)
    sinks = np.array([-np.inf, -3.0, 0.0, 2.5, 30.0, 1e4], np.float32)
    so, sl = _run_opt(p, scale, sinks=sinks)
    hq = 6
    sk = np.tile(sinks.astype(np.float64), out.shape[0] // hq)
    with np.errstate(over="ignore"):                 # a 1e4 sink: weight 0
        w = 1.0 / (1.0 + np.exp(sk - lse))
    np.testing.assert_allclose(so, out * w[:, None], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sl, np.logaddexp(lse, sk), rtol=1e-15, atol=1e-12)
    head0 = np.arange(out.shape[0]) % hq == 0       # sink -inf: no change
    np.testing.assert_array_equal(so[head0], out[head0])
    np.testing.assert_array_equal(sl[head0], lse[head0])
    with pytest.raises(ValueError):
        _run_opt(p, scale, sinks=sinks[:3])


def test_non_causal_matches_torch_brute_force():
    # a cached prefix attended in a pass of its own: every query of a
    # sequence sees all seq_len keys, seq_len may be below q_len, and a
    # sequence with no key gives out 0 and lse -inf
    rng = np.random.default_rng(34)
    p = _problem(rng, [6, 1, 3], [4, 30, 1], 4, 2, 64, 16)
    p["sl"][2] = 0
    scale = 0.125
    out, lse = _run_opt(p, scale, causal=False)
    ref, ref_lse = _sdpa_masked(p, scale, lambda L, ql: torch.ones(ql, L, dtype=torch.bool))
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)
    with pytest.raises(ValueError):
        _run_opt(p, scale, causal=False, window=4)


def test_prefix_pass_merged_with_new_keys_equals_one_causal_pass():
    # "shared/attention_kit.py", _attend_with_prefix: the chunk's queries
    # attend the cached prefix (all of it) and the new keys (causally) in two
    # passes, merged by log-sum-exp; here the prefix is whole pages, so the
    # new keys are the block table shifted by prefix / bs pages
    rng = np.random.default_rng(35)
    bs = 16
    prefix = [32, 0, 48]
    q_lens = [20, 7, 1]
    p = _problem(rng, q_lens, [a + b for a, b in zip(prefix, q_lens)], 4, 2, 64, bs)
    scale = 0.125
    full_out, full_lse = _run(p, scale)
    pre = dict(p, sl=np.array(prefix, np.int32))
    out_a, lse_a = _run_opt(pre, scale, causal=False)
    bt2 = np.full_like(p["bt"], -1)
    for s, P in enumerate(prefix):
        shifted = p["bt"][s, P // bs:]
        bt2[s, :shifted.shape[0]] = shifted
    new = dict(p, sl=np.array(q_lens, np.int32), bt=bt2)
    out_b, lse_b = _run(new, scale)
    out, lse = oracle.merge_states(out_a, lse_a, out_b, lse_b)
    np.testing.assert_allclose(out, full_out, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, full_lse, rtol=0, atol=1e-12)


def test_one_visible_key_gives_that_value_and_its_score():
    # "attention_impl.py" single-token path: a one-key softmax is exactly 1.
    rng = np.random.default_rng(2)
    p = _problem(rng, [1, 1], [1, 1], 4, 2, 64, 16)
    out, lse = _run(p, 0.2)
    qf = torch.from_numpy(p["q"].view(np.int16)).view(torch.bfloat16).double().numpy()
    for s in range(2):
        K = _gather(p, p["kc"], p["ks"], s, 1)[0]
        V = _gather(p, p["vc"], p["vs"], s, 1)[0]
        for h in range(4):
            r = s * 4 + h
            np.testing.assert_allclose(out[r], V[h // 2], rtol=0, atol=1e-15)
            # the softmax scale is an fp32 argument: 0.2 means float32(0.2)
            assert abs(lse[r] - float(np.float32(0.2)) * float(np.dot(qf[s, h], K[h // 2]))) < 1e-12


def test_zero_query_gives_mean_value_and_log_count():
    rng = np.random.default_rng(4)
    p = _problem(rng, [1, 4], [33, 20], 4, 2, 64, 16, q_scale=0.0)
    out, lse = _run(p, 0.3)
    out = out.reshape(-1, 4, 64)
    lse = lse.reshape(-1, 4)
    # decode row: 33 visible keys; prefill rows i = 0..3 see 16 + i + 1 keys
    for t, (s, n) in enumerate([(0, 33), (1, 17), (1, 18), (1, 19), (1, 20)]):
        V = _gather(p, p["vc"], p["vs"], s, n)
        for h in range(4):
            np.testing.assert_allclose(out[t, h], V[:, h // 2].mean(0), rtol=0, atol=1e-12)
            assert abs(lse[t, h] - math.log(n)) < 1e-12


def test_identical_keys_and_constant_values():
    # all keys equal -> uniform weights, lse = s + ln n; values constant per
    # channel -> output equals that constant (the weights sum to one)
    rng = np.random.default_rng(8)
    p = _problem(rng, [1, 3], [70, 45], 8, 2, 128, 16)
    p["kc"][:] = p["kc"][0, 0, 0][None, None, None, :]
    p["ks"][:] = p["ks"][0, 0, 0][None, None, None, :]
    p["vc"][:] = 7
    p["vs"][:] = _f16_bits_numpy(np.full(p["vs"].shape, 0.5))
    out, lse = _run(p, 0.1)
    qf = torch.from_numpy(p["q"].view(np.int16)).view(torch.bfloat16).double().numpy()
    k0 = _dequant(p["kc"][0, 0, 0], p["ks"][0, 0, 0])
    np.testing.assert_allclose(out, 3.5, rtol=0, atol=1e-12)
    counts = [70, 43, 44, 45]
    for t in range(4):
        for h in range(8):
            s0 = float(np.float32(0.1)) * float(np.dot(qf[t, h], k0))
            assert abs(lse[t * 8 + h] - (s0 + math.log(counts[t]))) < 1e-11


def test_gqa_head_h_reads_kv_head_h_over_qpk():
    rng = np.random.default_rng(6)
    hq, hk = 12, 3
    p = _problem(rng, [1], [40], hq, hk, 64, 16)
    for kv in range(hk):
        p["vc"][:, kv] = 10 * (kv + 1)
    p["vs"][:] = _f16_bits_numpy(np.full(p["vs"].shape, 1.0))
    out, _ = _run(p, 0.125)
    for h in range(hq):
        np.testing.assert_allclose(out[h], 10.0 * (h // (hq // hk) + 1), rtol=0, atol=1e-12)


def test_causal_limit_is_bottom_right_aligned():
    # value channel 0 of key j = j (code j, scale 1); q = 0 gives the mean of
    # the visible positions: query i of a chunk with context c sees 0..c+i
    rng = np.random.default_rng(7)
    L, ql = 100, 6
    p = _problem(rng, [ql], [L], 2, 1, 32, 16, q_scale=0.0)
    s = 0
    j = np.arange(L)
    blk = p["bt"][s, j // 16]
    p["vc"][blk, 0, 0, j % 16] = j.astype(np.int8)   # V pages are channel-major
    p["vs"][:] = _f16_bits_numpy(np.full(p["vs"].shape, 1.0))
    out, _ = _run(p, 1.0)
    out = out.reshape(ql, 2, 32)
    for i in range(ql):
        c = L - ql
        assert abs(out[i, 0, 0] - (c + i) / 2.0) < 1e-12


def test_paged_equals_contiguous():
    # the same logical cache laid out contiguously (identity block table) and
    # scattered (permuted table) gives the same result bit for bit
    rng = np.random.default_rng(10)
    p = _problem(rng, [3, 1], [45, 64], 4, 2, 64, 16, spare=0)
    out1, lse1 = _run(p, 0.125)
    # build the contiguous copy: sequence s page k -> physical block offset_s + k
    bt = p["bt"]
    pages = [(L + 15) // 16 for L in p["sl"]]
    ident = np.full_like(bt, -1)
    order = []
    pos = 0
    for s, n in enumerate(pages):
        ident[s, :n] = np.arange(pos, pos + n)
        order.extend(bt[s, :n].tolist())
        pos += n
    q = dict(p)
    for key in ("kc", "ks", "vc", "vs"):
        q[key] = np.ascontiguousarray(p[key][order])
    q["bt"] = ident
    out2, lse2 = _run(q, 0.125)
    np.testing.assert_array_equal(out1, out2)
    np.testing.assert_array_equal(lse1, lse2)


def test_split_segments_merged_by_lse_equal_one_joint_pass():
    rng = np.random.default_rng(12)
    p = _problem(rng, [1, 4], [300, 90], 4, 2, 64, 16)
    scale = 0.125
    full_out, full_lse = _run(p, scale)
    args = (p["q"], p["kc"], p["ks"], p["vc"], p["vs"], p["cu"], p["sl"], p["bt"], scale)
    for token, hi in ((0, 300), (3, 90)):
        for bounds in ([0, 150, 300], [0, 64, 128, 192, 256, 300], [0, 1, 300], [0, 300, 320]):
            parts = [oracle.attention_partial(*args, token=token, head=3, lo=a, hi=b)
                     for a, b in zip(bounds[:-1], bounds[1:])]
            m = [x[0] for x in parts]
            l = [x[1] for x in parts]
            acc = np.stack([x[2] for x in parts])
            out, lse = oracle.merge_partials(m, l, acc)
            r = token * 4 + 3
            np.testing.assert_allclose(out, full_out[r], rtol=0, atol=1e-12)
            assert abs(lse - full_lse[r]) < 1e-12


def test_merge_states_of_two_key_ranges_equals_one_joint_pass():
    # "shared/attention_kit.py" _merge_lse_: the attention over A and over B,
    # each normalized with its LSE, merge into the attention over A u B
    rng = np.random.default_rng(21)
    p = _problem(rng, [1, 3], [257, 64], 4, 2, 64, 16)
    scale = 0.125
    full_out, full_lse = _run(p, scale)
    args = (p["q"], p["kc"], p["ks"], p["vc"], p["vs"], p["cu"], p["sl"], p["bt"], scale)
    for token, n in ((0, 257), (2, 63), (3, 64)):
        for split in (1, 16, n // 2, n - 1):
            for head in (0, 3):
                a = oracle.attention_partial(*args, token=token, head=head, lo=0, hi=split)
                b = oracle.attention_partial(*args, token=token, head=head, lo=split, hi=n)
                out_a, lse_a = a[2] / a[1], a[0] + np.log(a[1])
                out_b, lse_b = b[2] / b[1], b[0] + np.log(b[1])
                out, lse = oracle.merge_states(out_a[None], [lse_a], out_b[None], [lse_b])
                r = token * 4 + head
                np.testing.assert_allclose(out[0], full_out[r], rtol=0, atol=1e-12)
                assert abs(lse[0] - full_lse[r]) < 1e-12


def test_merge_states_closed_forms():
    rng = np.random.default_rng(22)
    a = rng.standard_normal((5, 8))
    b = rng.standard_normal((5, 8))
    la = np.array([0.0, np.log(3.0), -np.inf, 2.0, -np.inf])
    lb = np.array([0.0, 0.0, 1.5, -np.inf, -np.inf])
    out, lse = oracle.merge_states(a, la, b, lb)
    np.testing.assert_allclose(out[0], (a[0] + b[0]) / 2, rtol=0, atol=1e-15)   # equal weights
    assert abs(lse[0] - np.log(2.0)) < 1e-15
    np.testing.assert_allclose(out[1], 0.75 * a[1] + 0.25 * b[1], rtol=0, atol=1e-15)  # 3 : 1
    assert abs(lse[1] - np.log(4.0)) < 1e-15
    np.testing.assert_array_equal(out[2], b[2])        # an empty side contributes nothing
    assert lse[2] == 1.5
    np.testing.assert_array_equal(out[3], a[3])
    assert lse[3] == 2.0
    np.testing.assert_array_equal(out[4], np.zeros(8))  # no key on either side
    assert lse[4] == -np.inf
    out2, lse2 = oracle.merge_states(b, lb, a, la)      # symmetric in its two parts
    np.testing.assert_allclose(out2, out, rtol=0, atol=1e-15)
    np.testing.assert_array_equal(lse2, lse)


def test_oracle_reports_bad_block_table():
    rng = np.random.default_rng(13)
    p = _problem(rng, [1], [40], 2, 1, 32, 16)
    p["bt"][0, 1] = p["kc"].shape[0] + 5
    with pytest.raises(RuntimeError):
        _run(p, 0.1)


# ----------------------------------------------------------------------------- fused norm + rotation store


def test_bf16_conversion_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(21)
    vals = [rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000)]
    # exact midpoints between neighbouring bf16 values (ties), normal and subnormal
    hb = np.arange(0, 0x7f7f, 13, dtype=np.uint32)
    lo = (hb << 16).view(np.float32).astype(np.float64)
    hi = ((hb + 1) << 16).view(np.float32).astype(np.float64)
    vals.append(((lo + hi) / 2).astype(np.float32))
    vals.append(np.array([0.0, 1e-40, 3.4e38, 3.3961776e38, np.inf, 1.00390625, 1.01171875],
                         np.float32))
    x = np.concatenate([np.asarray(v, np.float32) for v in vals])
    x = np.concatenate([x, -x])
    got = np.array([oracle.f32_to_bf16_bits(float(v)) for v in x], np.uint16)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(got, want)
    assert np.isnan(torch.tensor([oracle.f32_to_bf16_bits(float("nan"))], dtype=torch.int16)
                    .view(torch.bfloat16).float().item())


def _bf16_to_f64(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16) \
        .double().numpy()


def _rope_rows(rng, n, pairs, theta=None):
    ang = rng.uniform(-np.pi, np.pi, (n, pairs)) if theta is None else theta
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)


@pytest.mark.parametrize("d,scale", [(64, 3.0), (128, 3.0), (256, 3.0), (128, 1e-3)])
def test_rms_norm_matches_the_closed_form_within_bf16_rounding(d, scale):
    # y = x / sqrt(mean(x^2) + eps) * w: fp64 closed form against the oracle's
    # fp32 statistics and bf16 output (relative 2^-8 from the output rounding,
    # plus fp32 rounding of the statistics), with no systematic bias; at scale
    # 1e-3 eps is as large as the mean square
    rng = np.random.default_rng(22 + d)
    x = _bf16_bits(torch.from_numpy(rng.standard_normal((40, d)) * scale))
    w = _bf16_bits(torch.from_numpy(rng.uniform(0.2, 2.0, d)))
    eps = 1e-6
    got = oracle.norm_rope_rows(x, w, eps).astype(np.float64)
    xf, wf = _bf16_to_f64(x), _bf16_to_f64(w)
    want = xf / np.sqrt(np.mean(xf * xf, axis=1, keepdims=True) + eps) * wf
    assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) * (1 + 1e-5) + 1e-30)
    nz = want != 0
    assert abs(np.mean((got[nz] - want[nz]) / want[nz])) <= 2.0 ** -12
    # every value is a bf16 value (the norm output is rounded to the activation dtype)
    np.testing.assert_array_equal(
        _bf16_to_f64(_bf16_bits(torch.from_numpy(got))), got)


def test_rms_norm_is_exactly_scale_invariant_for_powers_of_two():
    # scaling a row by 2^k scales every fp32 step of the statistics exactly
    # (with eps 0): the normalized row is bit-identical
    rng = np.random.default_rng(23)
    x = _bf16_bits(torch.from_numpy(rng.standard_normal((16, 128))))
    w = _bf16_bits(torch.from_numpy(rng.uniform(0.5, 1.5, 128)))
    base = oracle.norm_rope_rows(x, w, 0.0)
    for k in (-6, 3, 9):
        xs = _bf16_bits(torch.from_numpy(_bf16_to_f64(x) * 2.0 ** k))
        np.testing.assert_array_equal(oracle.norm_rope_rows(xs, w, 0.0), base)


def test_no_norm_no_rotation_passes_the_values_through():
    rng = np.random.default_rng(24)
    x = _bf16_bits(torch.from_numpy(rng.standard_normal((8, 64))))
    np.testing.assert_array_equal(oracle.norm_rope_rows(x), _bf16_to_f64(x).astype(np.float32))


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotation_pairs_signs_and_identity(interleaved):
    rng = np.random.default_rng(25)
    n, d, rot = 6, 128, 96
    x = _bf16_bits(torch.from_numpy(rng.standard_normal((n, d))))
    y = _bf16_to_f64(x)
    # cos 1, sin 0: the identity, exactly
    ident = oracle.norm_rope_rows(x, rope_rows=_rope_rows(rng, n, rot // 2,
                                                          np.zeros((n, rot // 2))),
                                  interleaved=interleaved)
    np.testing.assert_array_equal(ident, y.astype(np.float32))
    # a quarter turn (cos 0, sin 1): lead <- -trail, trail <- lead, exactly;
    # the pairs are (p, p + rot/2), or (2p, 2p + 1) when interleaved
    quarter = np.stack([np.zeros((n, rot // 2)), np.ones((n, rot // 2))], -1).astype(np.float32)
    got = oracle.norm_rope_rows(x, rope_rows=quarter, interleaved=interleaved)
    p = np.arange(rot // 2)
    lead, trail = (2 * p, 2 * p + 1) if interleaved else (p, p + rot // 2)
    np.testing.assert_array_equal(got[:, lead], -y[:, trail])
    np.testing.assert_array_equal(got[:, trail], y[:, lead])
    np.testing.assert_array_equal(got[:, rot:], y[:, rot:])  # channels past rot unchanged


@pytest.mark.parametrize("interleaved", [False, True])
def test_rotation_matches_complex_multiplication(interleaved):
    # (y_lead + i y_trail) (cos + i sin) in fp64, within the fp32 rounding of
    # the page's fma form; every pair keeps its length
    rng = np.random.default_rng(26)
    n, d, rot = 50, 128, 128
    x = _bf16_bits(torch.from_numpy(rng.standard_normal((n, d)) * 4))
    rows = _rope_rows(rng, n, rot // 2)
    got = oracle.norm_rope_rows(x, rope_rows=rows, interleaved=interleaved).astype(np.float64)
    y = _bf16_to_f64(x)
    p = np.arange(rot // 2)
    lead, trail = (2 * p, 2 * p + 1) if interleaved else (p, p + rot // 2)
    z = (y[:, lead] + 1j * y[:, trail]) * (rows[..., 0].astype(np.float64)
                                           + 1j * rows[..., 1].astype(np.float64))
    bound = 2.0 ** -23 * (np.abs(y[:, lead]) + np.abs(y[:, trail])) * 2
    assert np.all(np.abs(got[:, lead] - z.real) <= bound)
    assert np.all(np.abs(got[:, trail] - z.imag) <= bound)


def test_fused_store_without_norm_or_rotation_is_kv_store():
    w = _small_store_problem(seed=5, hk=3, d=128, bs=32)
    k, v, slots = w.all_key_value()
    caches = []
    for fused in (False, True):
        kc, ks, vc, vs = [t.numpy() for t in inputs.empty_cache(w.num_blocks, 3, 32, 128)]
        ks, vs = ks.view(np.uint16), vs.view(np.uint16)
        if fused:
            assert oracle.kv_store_norm_rope(inputs.bf16_bits(k), inputs.bf16_bits(v),
                                             slots.numpy(), None, kc, ks, vc, vs) == 0
        else:
            oracle.kv_store(inputs.bf16_bits(k), inputs.bf16_bits(v), slots.numpy(), kc, ks, vc, vs)
        caches.append((kc, ks, vc, vs))
    for a, b in zip(*caches):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("interleaved", [False, True])
def test_fused_store_quantizes_each_tokens_rotated_row_at_its_slot(interleaved):
    # keys: normalized, rotated with the row of the token's own position, and
    # quantized from fp32 by the group quantizer (pinned above); values exactly
    # as kv_store stores them; a position outside the table skips the token
    rng = np.random.default_rng(27)
    hk, d, bs, n = 2, 128, 16, 40
    num_blocks = 4
    slots = rng.permutation(num_blocks * bs)[:n].astype(np.int64)
    slots[3] = -1
    positions = rng.integers(0, 300, n).astype(np.int64)
    positions[7] = 300  # past the table: skipped and counted
    table = _rope_rows(rng, 300, 32)  # rotary_dim 64 of 128
    k = _bf16_bits(torch.from_numpy(rng.standard_normal((n, hk, d)) * 2))
    v = _bf16_bits(torch.from_numpy(rng.standard_normal((n, hk, d))))
    wt = _bf16_bits(torch.from_numpy(rng.uniform(0.5, 1.5, d)))
    kc, ks, vc, vs = [t.numpy() for t in inputs.empty_cache(num_blocks, hk, bs, d)]
    ks, vs = ks.view(np.uint16), vs.view(np.uint16)
    bad = oracle.kv_store_norm_rope(k, v, slots, positions, kc, ks, vc, vs, wt, 1e-5, table,
                                    interleaved=interleaved)
    assert bad == 1
    vc_ref, vs_ref = [t.numpy() for t in inputs.empty_cache(num_blocks, hk, bs, d)][2:]
    vs_ref = vs_ref.view(np.uint16)
    kc_dummy, ks_dummy = [t.numpy() for t in inputs.empty_cache(num_blocks, hk, bs, d)][:2]
    keep = positions < 300
    oracle.kv_store(k[keep], v[keep], slots[keep], kc_dummy, ks_dummy.view(np.uint16), vc_ref,
                    vs_ref)
    np.testing.assert_array_equal(vc, vc_ref)
    np.testing.assert_array_equal(vs, vs_ref)
    for t in range(n):
        if slots[t] < 0 or not keep[t]:
            if slots[t] >= 0:
                assert np.all(kc[slots[t] // bs, :, slots[t] % bs] == -128)
            continue
        rows = oracle.norm_rope_rows(k[t], wt, 1e-5, np.repeat(table[positions[t]][None], hk, 0),
                                     interleaved=interleaved)
        for h in range(hk):
            for g in range(d // 32):
                codes, sbits = oracle.q8_quantize_group(rows[h, 32 * g:32 * g + 32])
                np.testing.assert_array_equal(kc[slots[t] // bs, h, slots[t] % bs,
                                                 32 * g:32 * g + 32], codes)
                assert ks[slots[t] // bs, h, slots[t] % bs, g] == sbits


# ----------------------------------------------------------------------------- fp8 keys, 4-bit values

V4_GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "v4_hand_examples.txt")


def _load_v4_golden():
    cases = []
    for line in open(V4_GOLDEN):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        name, xs, nib, sb, zb = [p.strip() for p in line.split(";")]
        x = np.array([float(v) for v in xs.split(",")], np.float32)
        cases.append((name, x, np.array([int(b, 16) for b in nib.split(",")], np.uint8),
                      int(sb, 16), int(zb, 16)))
    return cases


@pytest.mark.parametrize("case", _load_v4_golden(), ids=lambda c: c[0])
def test_v4_hand_examples(case):
    name, x, nib, sbits, zbits = case
    bits = _bf16_bits(torch.from_numpy(x))
    assert np.array_equal(_bf16_to_f64(bits), x.astype(np.float64))  # bf16-exact inputs
    got_nib, got_s, got_z = oracle.v4_quantize_rows(bits[None, :])
    np.testing.assert_array_equal(got_nib[0], nib)
    assert int(got_s[0]) == sbits and int(got_z[0]) == zbits


def test_e4m3_conversion_matches_torch_round_to_nearest_even():
    rng = np.random.default_rng(31)
    vals = [rng.standard_normal(3000) * 10.0 ** rng.uniform(-3, 2.6, 3000)]
    # midpoints between neighbouring e4m3 values (ties), normal and subnormal
    pos = np.arange(0, 0x7e, dtype=np.uint8)
    dec = torch.from_numpy(pos.copy()).view(torch.float8_e4m3fn).double().numpy()
    vals.append(((dec[:-1] + dec[1:]) / 2).astype(np.float32))
    vals.append(np.array([0.0, 448.0, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 1.0, 240.0, 464.0 - 1e-3],
                         np.float32))
    x = np.concatenate([np.asarray(v, np.float32) for v in vals])
    x = x[np.abs(x) < 464.0]  # where rounding to nearest stays at or below 448
    x = np.concatenate([x, -x])
    got = np.array([oracle.f32_to_e4m3_bits(float(v)) for v in x], np.uint8)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got, want)
    # saturation instead of NaN past the largest finite value
    for v in (464.0, 480.0, 1e6, float("inf")):
        assert oracle.f32_to_e4m3_bits(v) == 0x7e and oracle.f32_to_e4m3_bits(-v) == 0xfe


def test_e4m3_decode_matches_torch_for_every_pattern():
    bits = np.arange(256, dtype=np.uint16).astype(np.uint8)
    ref = torch.from_numpy(bits.copy()).view(torch.float8_e4m3fn).float().numpy()
    got = np.array([oracle.e4m3_bits_to_f32(int(b)) for b in bits], np.float32)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.all(np.isnan(got[~finite]))


def test_v4_invariants_on_random_rows():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((300, 128)) * 10.0 ** rng.uniform(-3, 2, (300, 1))
    x[::7] += rng.uniform(-50, 50, (x[::7].shape[0], 1))  # rows far from zero
    bits = _bf16_bits(torch.from_numpy(x))
    xf = _bf16_to_f64(bits)
    nib, sb, zb = oracle.v4_quantize_rows(bits)
    idx = np.stack([nib & 0xF, nib >> 4], -1).reshape(300, 128).astype(np.float64)
    s16 = sb.view(np.float16).astype(np.float64)[:, None]
    z16 = zb.view(np.float16).astype(np.float64)[:, None]
    lo, hi = xf.min(1, keepdims=True), xf.max(1, keepdims=True)
    s32 = (hi - lo) / 15
    # the row's min maps to 0 and its max to 15; a row that bf16 made constant
    # (small noise on a large offset) maps to 0 throughout
    flat = (hi == lo)[:, 0]
    assert 0 < flat.sum() < 300
    assert np.all(idx[np.arange(300), xf.argmin(1)] == 0)
    assert np.all(idx[~flat][np.arange((~flat).sum()), xf[~flat].argmax(1)] == 15)
    assert np.all(idx[flat] == 0)
    s32 = np.where(flat[:, None], 1e-8, s32)
    # each value within half a step of its code (plus fp32 rounding of the steps)
    assert np.all(np.abs(xf - (lo + idx * s32)) <= s32 * (0.5 + 1e-5))
    # round trip through the fp16 scale and zero: the fp16 rounding of both adds
    # at most 15 |s32 - s16| + |lo - z16|
    bound = s32 * 0.5 + 15 * np.abs(s32 - s16) + np.abs(lo - z16) + 1e-6 * s32
    assert np.all(np.abs(xf - (idx * s16 + z16)) <= bound)


def test_f8v4_store_places_each_tokens_row_at_its_slot():
    # what lands where: keys as e4m3 of each bf16 value (checked against torch's
    # conversion), values as the row quantizer's nibbles, read back at
    # (slot / bs, head, slot % bs) with the channel-major nibble layout
    hk, d, bs = 3, 64, 16
    rng = np.random.default_rng(33)
    n_tok, num_blocks = 45, 5
    slots = rng.permutation(num_blocks * bs)[:n_tok].astype(np.int64)
    slots[[2, 17]] = -1
    k = _bf16_bits(torch.from_numpy(rng.standard_normal((n_tok, hk, d)) * 10.0 ** (np.arange(hk) - 1)[None, :, None]))
    v = _bf16_bits(torch.from_numpy(rng.standard_normal((n_tok, hk, d)) * 3.0 ** np.arange(hk)[None, :, None]))
    shapes = oracle.f8v4_cache_shapes(num_blocks, hk, bs, d)
    kc = np.full(shapes[0], 0xff, np.uint8)
    vc = np.full(shapes[1], 0xff, np.uint8)
    vs = np.full(shapes[2], 0xffff, np.uint16)
    vz = np.full(shapes[3], 0xffff, np.uint16)
    assert oracle.kv_store_f8v4(k, v, slots, kc, vc, vs, vz) == 0
    for t in range(n_tok):
        if slots[t] < 0:
            continue
        blk, off = slots[t] // bs, slots[t] % bs
        for h in range(hk):
            want_k = torch.from_numpy(_bf16_to_f64(k[t, h]).astype(np.float32)).to(
                torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(kc[blk, h, off], want_k)
            nib, sb, zb = oracle.v4_quantize_rows(v[t, h][None])
            idx = np.stack([nib[0] & 0xF, nib[0] >> 4], -1).reshape(d)
            got = (vc[blk, h, :, off // 2] >> (4 * (off % 2))) & 0xF
            np.testing.assert_array_equal(got, idx)
            assert vs[blk, h, off] == sb[0] and vz[blk, h, off] == zb[0]
    written = np.zeros(num_blocks * bs, bool)
    written[slots[slots >= 0]] = True
    unw = np.nonzero(~written)[0]
    assert np.all(kc[unw // bs, :, unw % bs] == 0xff)
    assert np.all(vs[unw // bs, :, unw % bs] == 0xffff)


def test_attention_over_f8v4_cache_matches_torch_sdpa():
    # brute force on the dequantized values (e4m3 keys; idx * scale + zero values)
    # with torch's fp64 scaled_dot_product_attention and an explicit causal mask
    rng = np.random.default_rng(34)
    hq, hk, d, bs = 4, 2, 64, 16
    q_lens, seq_lens = [5, 1, 3], [21, 40, 3]
    S = 3
    pages = [(L + bs - 1) // bs for L in seq_lens]
    num_blocks = sum(pages) + 2
    perm = rng.permutation(num_blocks).astype(np.int32)
    bt = np.full((S, max(pages)), -1, np.int32)
    pos = 0
    for s, n in enumerate(pages):
        bt[s, :n] = perm[pos:pos + n]
        pos += n
    cu = np.zeros(S + 1, np.int32)
    cu[1:] = np.cumsum(q_lens)
    T = int(cu[-1])
    shapes = oracle.f8v4_cache_shapes(num_blocks, hk, bs, d)
    kc = rng.integers(0, 256, shapes[0]).astype(np.uint8)
    kc[(kc & 0x7f) == 0x7f] = 0x3c  # no NaN patterns
    vc = rng.integers(0, 256, shapes[1]).astype(np.uint8)
    vs = np.asarray(rng.uniform(0.01, 0.2, shapes[2]), np.float16).view(np.uint16)
    vz = np.asarray(rng.uniform(-1, 1, shapes[3]), np.float16).view(np.uint16)
    qb = _bf16_bits(torch.from_numpy(rng.standard_normal((T, hq, d))))
    scale = d ** -0.5
    out, lse = oracle.paged_attention(qb, kc, None, vc, vs, cu, np.array(seq_lens, np.int32),
                                      bt, scale, v_zero=vz)
    kdeq = torch.from_numpy(kc.copy()).view(torch.float8_e4m3fn).double().numpy()
    idx = np.stack([vc & 0xF, vc >> 4], -1).reshape(num_blocks, hk, d, bs)
    vdeq = idx * vs.view(np.float16).astype(np.float64)[:, :, None, :] + \
        vz.view(np.float16).astype(np.float64)[:, :, None, :]      # [nb, hk, d, bs]
    qf = _bf16_to_f64(qb)
    for s in range(S):
        L, ql = seq_lens[s], q_lens[s]
        j = np.arange(L)
        K = kdeq[bt[s, j // bs], :, j % bs, :]                  # [L, hk, d]
        V = vdeq[bt[s, j // bs], :, :, j % bs]                  # [L, hk, d]
        qs = torch.from_numpy(qf[cu[s]:cu[s + 1]]).transpose(0, 1)          # [hq, ql, d]
        Kt = torch.from_numpy(K).transpose(0, 1).repeat_interleave(hq // hk, 0)
        Vt = torch.from_numpy(V).transpose(0, 1).repeat_interleave(hq // hk, 0)
        mask = torch.from_numpy(np.arange(L)[None, :] <= (L - ql + np.arange(ql))[:, None])
        ref = torch.nn.functional.scaled_dot_product_attention(qs, Kt, Vt, attn_mask=mask,
                                                               scale=scale)
        sc = (qs @ Kt.transpose(1, 2)) * scale
        ref_lse = torch.logsumexp(sc.masked_fill(~mask, float("-inf")), -1)
        rows = (np.arange(cu[s], cu[s + 1])[:, None] * hq + np.arange(hq)[None, :]).T
        np.testing.assert_allclose(out[rows.reshape(-1)].reshape(hq, ql, d), ref.numpy(),
                                   rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(lse[rows.reshape(-1)].reshape(hq, ql), ref_lse.numpy(),
                                   rtol=1e-12, atol=1e-12)

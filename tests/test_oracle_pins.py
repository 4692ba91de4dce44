"""Pins for the fp64 CPU oracle: closed forms, invariants, a textbook reduction
and brute force on tiny inputs.  Each test states which part of the definition
(gfx950 'Unified paged attention on gfx950, from the math up', section 1) a
plausible mistake in the oracle would break.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from paged_varlen_flash_gb300 import workloads as W
from tests.helpers import (decode_tag, gather_logical, position_tags, scatter_logical,
                           tag_values, token_of_row)

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "micro_examples.json")


def _run(w, **over):
    kw = dict(causal=w.causal, softcap=w.softcap, window=w.window,
              alibi_slopes=w.alibi_slopes, sinks=w.sinks)
    kw.update(over)
    return oracle.forward(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                          w.seqused_k, w.scale, **kw)


def _blank(seqlens_q, seqlens_k, hq=4, hk=2, d=64, b=16, seed=0, **kw):
    need = sum((k + b - 1) // b for k in seqlens_k)
    return W.build("pin", hq, hk, d, b, seqlens_q, seqlens_k, need + 3, 1.0 / math.sqrt(d),
                   seed=seed, values=False, poison=True, bt_pad=1, **kw)


def _visible_range(i, ctx, sk, causal, window):
    hi = i + ctx if causal else sk - 1
    lo = max(0, i + ctx - window + 1) if window > 0 else 0
    return lo, hi


# --------------------------------------------------------------------------
# Closed form: constant keys -> O = mean of the visible V rows.
# Pins the causal / window edges, ctx = S_k - S_q, the paged lookup and the
# normalisation (a dropped or extra key, a wrong ctx or a wrong block changes
# the mean of the position tags).
# --------------------------------------------------------------------------
@pytest.mark.parametrize("causal,window", [(True, 0), (True, 7), (True, 1), (False, 0),
                                           (True, 200)])
def test_constant_keys_give_mean_of_visible_values(causal, window):
    sq = [5, 16, 1, 33]
    sk = [37, 16, 50, 90]
    w = _blank(sq, sk, causal=causal, window=window, seed=3)
    g = torch.Generator().manual_seed(5)
    w.q = torch.randn(w.total_q, w.hq, w.d, generator=g).to(torch.bfloat16)
    kl, vl = [], []
    c = torch.randn(w.hk, w.d, generator=g)
    for s in range(w.num_seqs):
        kl.append(c.expand(sk[s], w.hk, w.d).clone())
        vl.append(position_tags(sk[s], w.hk, w.d))
    scatter_logical(w, kl, vl)
    out = _run(w)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        lo, hi = _visible_range(i, ctx, sk[s], causal, window)
        js = np.arange(lo, hi + 1, dtype=np.int64)
        for h in range(w.hq):
            o = out[tok, h]
            tags = tag_values(js, h // w.g)
            for k in range(4):
                assert abs(o[k] - np.mean(tags[k])) < 1e-12
            assert np.all(o[4:] == 0)


def test_window_of_one_returns_the_diagonal_value():
    """W = 1 keeps only key i + ctx, so O = V_{i+ctx} whatever the logits are
    (the page-literal reading that keeps W + 1 keys would average two rows)."""
    sq = [4, 9, 1]
    sk = [20, 9, 33]
    w = _blank(sq, sk, window=1, seed=4)
    g = torch.Generator().manual_seed(6)
    w.q = torch.randn(w.total_q, w.hq, w.d, generator=g).to(torch.bfloat16)
    kl = [torch.randn(k, w.hk, w.d, generator=g) for k in sk]
    vl = [position_tags(k, w.hk, w.d) for k in sk]
    scatter_logical(w, kl, vl)
    out = _run(w)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        for h in range(w.hq):
            assert decode_tag(out[tok, h]) == (i + ctx, h // w.g)
            assert abs(out[tok, h, 3] - tag_values(i + ctx, h // w.g)[3]) < 1e-12


# --------------------------------------------------------------------------
# One dominant key per (row, kv head): O = V_target to far below bf16 ulp.
# Pins the GQA head map, the token -> sequence map and the paged lookup.
# --------------------------------------------------------------------------
def test_dominant_key_selects_its_value_row():
    sq = [7, 30, 1]
    sk = [40, 30, 77]
    w = _blank(sq, sk, hq=8, hk=2, seed=8)
    w.scale = 1.0
    q = torch.zeros(w.total_q, w.hq, w.d)
    kl = [torch.zeros(k, w.hk, w.d) for k in sk]
    g = torch.Generator().manual_seed(9)
    targets = {}
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        q[tok, :, i] = 1.0
        for hkv in range(w.hk):
            t = int(torch.randint(0, i + ctx + 1, (1,), generator=g))
            targets[(tok, hkv)] = t
            kl[s][t, hkv, i] = 64.0
    w.q = q.to(torch.bfloat16)
    scatter_logical(w, kl, [position_tags(k, w.hk, w.d) for k in sk])
    out = _run(w)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        for h in range(w.hq):
            t = targets[(tok, h // w.g)]
            assert decode_tag(out[tok, h]) == (t, h // w.g)
            assert abs(out[tok, h, 0] - tag_values(t, h // w.g)[0]) < 1e-9


# --------------------------------------------------------------------------
# Sinks: with K = 0 every logit is 0, so a sink of ln(m n) gives
# O = mean(V) / (1 + m); +inf gives 0; -inf is the same as no sink.
# --------------------------------------------------------------------------
def test_sink_closed_forms():
    n = 45
    w = _blank([1], [n], hq=4, hk=1, seed=10)
    g = torch.Generator().manual_seed(11)
    w.q = torch.randn(1, w.hq, w.d, generator=g).to(torch.bfloat16)
    scatter_logical(w, [torch.zeros(n, 1, w.d)], [position_tags(n, 1, w.d)])
    mean0 = np.mean(tag_values(np.arange(n), 0)[0])
    sinks = torch.tensor([math.log(n * (h + 1)) for h in range(w.hq)], dtype=torch.float64)
    out = _run(w, sinks=sinks)
    for h in range(w.hq):
        assert abs(out[0, h, 0] - mean0 / (h + 2)) < 1e-12
    inf = _run(w, sinks=torch.full((w.hq,), math.inf, dtype=torch.float64))
    assert np.all(inf == 0.0)
    ninf = _run(w, sinks=torch.full((w.hq,), -math.inf, dtype=torch.float64))
    assert np.array_equal(ninf, _run(w, sinks=None))


# --------------------------------------------------------------------------
# Softcap: c -> 0 flattens every logit (O -> mean of visible V); c -> inf is
# the identity; and a tiny cap applied before ALiBi leaves pure ALiBi weights
# (if ALiBi came first the tiny cap would flatten it too).
# --------------------------------------------------------------------------
def _random_kv(w, seed):
    g = torch.Generator().manual_seed(seed)
    w.q = torch.randn(w.total_q, w.hq, w.d, generator=g).to(torch.bfloat16)
    kl = [torch.randn(k, w.hk, w.d, generator=g) for k in w.seqlens_k]
    vl = [position_tags(k, w.hk, w.d) for k in w.seqlens_k]
    scatter_logical(w, kl, vl)


def test_softcap_limits():
    sq, sk = [6, 3], [40, 70]
    w = _blank(sq, sk, seed=12)
    _random_kv(w, 13)
    tiny = _run(w, softcap=1e-9)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        js = np.arange(0, i + ctx + 1)
        for h in range(w.hq):
            assert abs(tiny[tok, h, 0] - np.mean(tag_values(js, 0)[0])) < 1e-6
    big = _run(w, softcap=1e12)
    base = _run(w, softcap=0.0)
    assert np.max(np.abs(big - base)) < 1e-10


def _geometric_mean_index(lo, n, a):
    """Mean of j over j = lo .. lo+n-1 under weights e^{a j} (closed form of a
    geometric series)."""
    r = math.exp(a)
    return lo + r / (1 - r) - n * r ** n / (1 - r ** n)


@pytest.mark.parametrize("window", [0, 9])
def test_alibi_closed_form_and_order_after_softcap(window):
    sq, sk = [3, 1], [60, 25]
    w = _blank(sq, sk, hq=4, hk=2, window=window, seed=14)
    slopes = torch.tensor([0.5, 0.25, 0.125, 0.0625], dtype=torch.float64)
    g = torch.Generator().manual_seed(15)
    w.q = torch.randn(w.total_q, w.hq, w.d, generator=g).to(torch.bfloat16)
    vl = [position_tags(k, w.hk, w.d) for k in sk]
    # K = 0: logits are exactly slope * (j - ctx).
    scatter_logical(w, [torch.zeros(k, w.hk, w.d) for k in sk], vl)
    out0 = _run(w, alibi_slopes=slopes)
    # Random K but a vanishing cap applied first: the same ALiBi-only weights.
    scatter_logical(w, [torch.randn(k, w.hk, w.d, generator=g) for k in sk], vl)
    out1 = _run(w, alibi_slopes=slopes, softcap=1e-9)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        lo, hi = _visible_range(i, ctx, sk[s], True, window)
        for h in range(w.hq):
            want = _geometric_mean_index(lo, hi - lo + 1, float(slopes[h])) + 1  # tag = j + 1
            assert abs(out0[tok, h, 0] - want) < 1e-9
            assert abs(out1[tok, h, 0] - want) < 1e-6


# --------------------------------------------------------------------------
# Invariants.
# --------------------------------------------------------------------------
def _flagged_random(seed, **kw):
    w = W.random_small(seed, num_seqs=4, hq=8, hk=2, d=64, b=16, sq=(1, 30),
                       ctx=(0, 60), **kw)
    return w


def test_weights_sum_to_one_and_reproduce_the_output():
    w = _flagged_random(20, softcap=5.0, window=17, sinks=True, alibi=True)
    for tok in range(0, w.total_q, 7):
        for h in (0, 3, 7):
            wt, o = oracle.row_weights(w.q, w.k_cache, w.v_cache, w.block_table,
                                       w.cu_seqlens_q, w.seqused_k, w.scale, tok, h,
                                       causal=True, softcap=5.0, window=17,
                                       alibi_slopes=w.alibi_slopes, sinks=w.sinks)
            assert abs(wt.sum() - 1.0) < 1e-12
            assert np.all(wt >= 0)
            s, i, ctx = token_of_row(w)[tok]
            lo, hi = _visible_range(i, ctx, w.seqlens_k[s], True, 17)
            assert np.all(wt[:lo] == 0) and np.all(wt[hi + 1:-1] == 0)
            vl = gather_logical(w, w.v_cache, s)[:, h // w.g].double().numpy()
            assert np.max(np.abs(wt[:-1] @ vl - o)) < 1e-12


def test_block_permutation_leaves_output_unchanged():
    w = _flagged_random(21, softcap=30.0, sinks=True)
    base = _run(w)
    g = torch.Generator().manual_seed(22)
    perm = torch.randperm(w.num_blocks, generator=g)
    k2 = torch.empty_like(w.k_cache)
    v2 = torch.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt = w.block_table.clone()
    used = bt >= 0
    bt[used] = perm[bt[used].long()].to(torch.int32)
    w.k_cache, w.v_cache, w.block_table = k2, v2, bt
    assert np.array_equal(_run(w), base)


def test_chunk_rows_equal_full_prefill_rows():
    L, m = 70, 23
    full = _blank([L], [L], seed=23)
    _random_kv(full, 24)
    chunk = _blank([m], [L], seed=23)
    chunk.k_cache, chunk.v_cache, chunk.block_table = full.k_cache, full.v_cache, full.block_table
    chunk.q = full.q[L - m:].clone()
    a = _run(full)[L - m:]
    b = _run(chunk)
    assert np.array_equal(a, b)


def test_gqa_equals_replicated_mha():
    w = _flagged_random(25, sinks=True, alibi=True, window=11)
    gqa = _run(w)
    rep = W.build("rep", w.hq, w.hq, w.d, w.b, w.seqlens_q, w.seqlens_k, w.num_blocks,
                  w.scale, values=False, poison=False)
    rep.q = w.q
    rep.block_table = w.block_table
    rep.k_cache = w.k_cache.repeat_interleave(w.g, dim=2)
    rep.v_cache = w.v_cache.repeat_interleave(w.g, dim=2)
    mha = _run(rep, alibi_slopes=w.alibi_slopes, sinks=w.sinks, window=11)
    assert np.array_equal(gqa, mha)


def test_window_wider_than_context_is_no_window():
    w = _flagged_random(26)
    assert np.array_equal(_run(w, window=10 ** 6), _run(w, window=0))


# --------------------------------------------------------------------------
# Textbook reduction: S_q = S_k, one block, identity table -> ordinary causal
# scaled-dot-product attention, here torch's fp64 math on the CPU.
# --------------------------------------------------------------------------
@pytest.mark.parametrize("hq,hk,causal", [(2, 2, True), (6, 2, True), (4, 4, False)])
def test_reduces_to_textbook_sdpa(hq, hk, causal):
    S, d = 48, 64
    w = W.build("sdpa", hq, hk, d, S, [S], [S], 1, 1.0 / math.sqrt(d), seed=27,
                causal=causal, poison=False, block_ids=torch.tensor([0]))
    out = _run(w)
    q = w.q.double().permute(1, 0, 2)                    # [hq, S, d]
    k = w.k_cache[0].double().permute(1, 0, 2)           # [hk, S, d]
    v = w.v_cache[0].double().permute(1, 0, 2)
    k = k.repeat_interleave(hq // hk, dim=0)
    v = v.repeat_interleave(hq // hk, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(
        q, k, v, is_causal=causal, scale=w.scale).permute(1, 0, 2).numpy()
    assert np.max(np.abs(out - ref)) < 1e-12


# --------------------------------------------------------------------------
# Brute force with a different algorithm: the streaming (m, l, o) recurrence
# over random key tiles (gfx1151 ALGORITHM.md section 3) and random split
# points merged by re-basing to the global max (gfx950 ALGORITHM.md section 5)
# reach the same rows as the oracle's direct evaluation.
# --------------------------------------------------------------------------
def _streamed_row(logits, vrows, sink, rng):
    n = len(logits)
    cuts = sorted(set(rng.integers(0, n + 1, size=rng.integers(0, 4)).tolist()) | {0, n})
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        m, l, o = -np.inf, 0.0, np.zeros(vrows.shape[1])
        t = a
        while t < b:
            e = min(b, t + int(rng.integers(1, 9)))
            s_t = logits[t:e]
            m_new = max(m, np.max(s_t)) if e > t else m
            if m_new == -np.inf:
                t = e
                continue
            alpha = math.exp(m - m_new) if m > -np.inf else 0.0
            p = np.exp(s_t - m_new)
            l = alpha * l + p.sum()
            o = alpha * o + p @ vrows[t:e]
            m = m_new
            t = e
        parts.append((m, l, o))
    M = max([p[0] for p in parts] + [sink])
    if M == -np.inf:
        return np.zeros(vrows.shape[1])
    L = sum(math.exp(p[0] - M) * p[1] for p in parts if p[0] > -np.inf)
    O = sum(math.exp(p[0] - M) * p[2] for p in parts if p[0] > -np.inf)
    if sink > -np.inf:
        L += math.exp(sink - M)
    return O / L if L > 0 else np.zeros(vrows.shape[1])


@pytest.mark.parametrize("seed", [30, 31, 32])
def test_streaming_and_split_merge_agree_with_direct_rows(seed):
    w = _flagged_random(seed, softcap=8.0, window=13, sinks=True, alibi=True)
    out = _run(w)
    rng = np.random.default_rng(seed)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        K = gather_logical(w, w.k_cache, s).double().numpy()
        V = gather_logical(w, w.v_cache, s).double().numpy()
        for h in range(w.hq):
            hk = h // w.g
            x = w.scale * (K[:, hk] @ w.q[tok, h].double().numpy())
            x = 8.0 * np.tanh(x / 8.0)
            x = x + float(w.alibi_slopes[h]) * (np.arange(len(x)) - ctx)
            lo, hi = _visible_range(i, ctx, len(x), True, 13)
            logits = x[lo:hi + 1]
            row = _streamed_row(logits, V[lo:hi + 1, hk], float(w.sinks[h]), rng)
            assert np.max(np.abs(row - out[tok, h])) < 1e-12


# --------------------------------------------------------------------------
# Hand-derived worked examples (tests/golden/micro_examples.json).
# --------------------------------------------------------------------------
def golden_cases():
    with open(GOLDEN) as f:
        return json.load(f)["cases"]


def golden_workload(case):
    sq, sk = case["seqlens_q"], case["seqlens_k"]
    w = W.build(case["name"], case["hq"], case["hk"], case["d"], case["b"], sq, sk,
                sum((k + case["b"] - 1) // case["b"] for k in sk) + 2, case["scale"],
                seed=0, values=False, poison=True, causal=case["causal"],
                softcap=case["softcap"], window=case["window"])
    q = torch.zeros(w.total_q, w.hq, w.d)
    for tok, h, dim, val in case["q"]:
        q[tok, h, dim] = val
    kl = [torch.zeros(k, w.hk, w.d) for k in sk]
    vl = [torch.zeros(k, w.hk, w.d) for k in sk]
    for s, j, hk, dim, val in case["k"]:
        kl[s][j, hk, dim] = val
    for s, j, hk, dim, val in case["v"]:
        vl[s][j, hk, dim] = val
    w.q = q.to(torch.bfloat16)
    scatter_logical(w, kl, vl)
    if case["sinks"] is not None:
        w.sinks = torch.tensor(case["sinks"], dtype=torch.float64)
    if case["alibi"] is not None:
        w.alibi_slopes = torch.tensor(case["alibi"], dtype=torch.float64)
    expected = np.zeros((w.total_q, w.hq, w.d))
    for tok, h, dim, val in case["expected"]:
        expected[tok, h, dim] = val
    return w, expected


@pytest.mark.parametrize("case", golden_cases(), ids=lambda c: c["name"])
def test_golden_micro_examples(case):
    w, expected = golden_workload(case)
    assert np.max(np.abs(_run(w) - expected)) < 1e-12


# --------------------------------------------------------------------------
# Malformed inputs and degenerate shapes.
# --------------------------------------------------------------------------
def test_rejects_context_shorter_than_chunk_and_bad_blocks():
    w = _blank([5], [5], seed=40)
    w.seqused_k = torch.tensor([4], dtype=torch.int32)
    with pytest.raises(oracle.OracleError) as e:
        _run(w)
    assert e.value.code == -2
    w = _blank([5], [5], seed=40)
    w.block_table[0, 0] = w.num_blocks
    with pytest.raises(oracle.OracleError) as e:
        _run(w)
    assert e.value.code == -3


def test_empty_sequences_and_zero_context():
    w = _blank([0, 3, 0], [0, 3, 9], seed=41)
    _random_kv(w, 42)
    out = _run(w)
    assert out.shape == (3, w.hq, w.d)
    assert np.all(np.isfinite(out))
    # First row of a self-attention sequence sees only key 0: O = V_0.
    V0 = gather_logical(w, w.v_cache, 1)[0].double().numpy()
    for h in range(w.hq):
        assert np.max(np.abs(out[0, h] - V0[h // w.g])) < 1e-12


def test_sampled_rows_match_full_forward():
    w = _flagged_random(43, softcap=20.0, sinks=True, window=25)
    full = _run(w)
    ids = W.sample_rows(w, 40, seed=1)
    part = oracle.forward_workload(w, row_ids=ids)
    flat = full.reshape(-1, w.d)
    assert np.array_equal(part, flat[ids.numpy()])


# ---------------------------------------------------------------------------
# fp8 e4m3 KV cache (gfx950 page, section 7.3): decoder, scales.
# ---------------------------------------------------------------------------

def test_e4m3_decoder_matches_torch_for_every_code():
    """The oracle's e4m3 decoder equals PyTorch's float8_e4m3fn -> fp32
    conversion (an independent implementation of the OCP format) on all 256
    codes, NaN codes included."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_value(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])
    assert np.array_equal(np.signbit(got[ok]), np.signbit(ref[ok]))
    # A few values the format fixes by hand: 1, the largest finite, the
    # smallest subnormal and the smallest normal.
    assert oracle.e4m3_value(0x38) == 1.0 and oracle.e4m3_value(0x7E) == 448.0
    assert oracle.e4m3_value(0x01) == 2.0 ** -9 and oracle.e4m3_value(0x08) == 2.0 ** -6


def _decoded_bf16(codes, scale):
    """e4m3 codes (uint8) -> bf16 tensor of code * scale (exact for these scales)."""
    return (codes.view(torch.float8_e4m3fn).to(torch.float32) * scale).to(torch.bfloat16)


@pytest.mark.parametrize("flags", [dict(), dict(softcap=20.0, sinks=True), dict(alibi=True, window=9)])
def test_fp8_cache_equals_attention_on_decoded_values(flags):
    """fp8 K/V with power-of-two scales: every decoded value times its scale is
    exact in bf16, so the fp8 oracle must equal the bf16 oracle on the decoded
    caches (pins the decode, the scale on each tensor and the paging)."""
    w = W.random_small(11, hq=8, hk=2, d=64, kv_fp8=True, kv_scale=0.125, **flags)
    kw = dict(causal=w.causal, softcap=w.softcap, window=w.window,
              alibi_slopes=w.alibi_slopes, sinks=w.sinks)
    got = oracle.forward(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                         w.seqused_k, w.scale, k_scale=0.125, v_scale=0.25, **kw)
    kb = _decoded_bf16(w.k_cache, 0.125)
    vb = _decoded_bf16(w.v_cache, 0.25)
    want = oracle.forward(w.q, kb, vb, w.block_table, w.cu_seqlens_q, w.seqused_k,
                          w.scale, **kw)
    assert not np.isnan(got).any()
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def test_fp8_scales_fold_into_tau_and_the_output():
    """k_scale multiplies every logit before the score chain, so it can move into
    tau; v_scale multiplies every value row, so it scales O."""
    w = W.random_small(12, hq=4, hk=1, d=64, kv_fp8=True, kv_scale=1.0, softcap=15.0)
    args = (w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q, w.seqused_k)
    kw = dict(causal=True, softcap=w.softcap)
    a = oracle.forward(*args, w.scale, k_scale=0.3, v_scale=1.0, **kw)
    b = oracle.forward(*args, w.scale * 0.3, k_scale=1.0, v_scale=1.0, **kw)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-12)
    c = oracle.forward(*args, w.scale, k_scale=0.3, v_scale=3.0, **kw)
    np.testing.assert_allclose(c, 3.0 * a, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# QQ-bias (gfx950 page, section 1 step 4): s_j += bias[i, j - ctx] for keys
# inside the query section (j >= ctx), after softcap / ALiBi, before the masks.
# ---------------------------------------------------------------------------

def _constant_key_workload(sq, sk, causal=True, softcap=0.0, seed=21):
    """Constant keys (every logit equal) and position-tag values."""
    w = _blank(sq, sk, causal=causal, seed=seed, softcap=softcap)
    g = torch.Generator().manual_seed(seed + 1)
    w.q = torch.randn(w.total_q, w.hq, w.d, generator=g).to(torch.bfloat16)
    c = torch.randn(w.hk, w.d, generator=g)
    scatter_logical(w, [c.expand(k, w.hk, w.d).clone() for k in sk],
                    [position_tags(k, w.hk, w.d) for k in sk])
    return w


@pytest.mark.parametrize("causal", [True, False])
def test_qq_bias_closed_form_on_constant_keys(causal):
    """Equal logits: key j of row i gets weight e^{bias[i, j - ctx]} inside the
    query section and 1 before it, so O is the weighted mean of the visible
    position tags -- pins the (i, j - ctx) indexing, the section boundary and
    the natural-log domain."""
    sq, sk = [6, 1, 9], [20, 5, 9]
    w = _constant_key_workload(sq, sk, causal=causal)
    g = torch.Generator().manual_seed(3)
    bias = torch.randn(12, 12, generator=g, dtype=torch.float64)
    bias[2, 1] = -math.inf     # drops one key of local row 2 exactly
    out = _run(w, qq_bias=bias)
    bnp = bias.numpy()
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        lo, hi = _visible_range(i, ctx, sk[s], causal, 0)
        js = np.arange(lo, hi + 1, dtype=np.int64)
        wt = np.array([math.exp(bnp[i, j - ctx]) if j >= ctx else 1.0 for j in js])
        for h in range(w.hq):
            tags = tag_values(js, h // w.g)
            for k in range(4):
                want = float(np.sum(wt * np.asarray(tags[k], dtype=np.float64)) / np.sum(wt))
                assert abs(out[tok, h, k] - want) < 1e-12


def test_qq_bias_zero_is_no_bias_and_it_is_added_after_softcap():
    w = _constant_key_workload([7, 3], [12, 3], softcap=0.5)
    base = _run(w)
    np.testing.assert_array_equal(_run(w, qq_bias=np.zeros((8, 8))), base)
    # A bias of 2 in the query section multiplies those keys' weights by e^2
    # whatever the cap; had the bias gone through tanh, the cap of 0.5 would
    # have flattened it to at most e^0.5.
    wts = oracle.row_weights(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                             w.seqused_k, w.scale, token=4, head=1, softcap=0.5)[0]
    wtb = oracle.row_weights(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                             w.seqused_k, w.scale, token=4, head=1, softcap=0.5,
                             qq_bias=np.full((8, 8), 2.0))[0]
    ctx = 12 - 7
    manual = wts[:-1].copy()
    manual[ctx:] *= math.exp(2.0)
    manual /= manual.sum()
    np.testing.assert_allclose(wtb[:-1], manual, rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------------------
# Sparse top-k mode ("[Triton/Gluon] [GFX950] Sparse paged attention and Sparse
# MLA": each query token attends to its own list of key positions).
# ---------------------------------------------------------------------------

def _full_lists(w, permute_seed=None):
    """Every key of each token's sequence, in order (or permuted per token)."""
    kmax = max(w.seqlens_k)
    rows, lens = [], []
    g = torch.Generator().manual_seed(permute_seed or 0)
    for s, i, ctx in token_of_row(w):
        sk = w.seqlens_k[s]
        pos = torch.arange(sk, dtype=torch.int32)
        if permute_seed is not None:
            pos = pos[torch.randperm(sk, generator=g)]
        row = torch.full((kmax,), -1, dtype=torch.int32)
        row[:sk] = pos
        rows.append(row)
        lens.append(sk)
    return torch.stack(rows), torch.tensor(lens, dtype=torch.int32)


@pytest.mark.parametrize("flags", [{}, dict(softcap=5.0, alibi=True, sinks=True, window=13),
                                   dict(causal=False, qq_bias=True), dict(sinks=True, qq_bias=True)])
def test_topk_list_of_every_key_in_order_is_the_dense_definition(flags):
    """A list holding keys 0 .. S_k-1 in order takes exactly the dense row's
    sum in the dense row's order: identical outputs, so the list mode applies
    the same score chain and masks with j = the listed position."""
    w = _flagged_random(60, **flags)
    qq = {"qq_bias": w.qq_bias} if w.qq_bias is not None else {}
    idx, lens = _full_lists(w)
    assert np.array_equal(_run(w, topk_idx=idx, topk_len=lens, **qq), _run(w, **qq))


def test_topk_list_order_does_not_matter():
    """A per-token permutation of the full list changes only the summation
    order: catches a weight or value taken from the entry index instead of the
    listed position."""
    w = _flagged_random(61, softcap=5.0, alibi=True, sinks=True)
    idx, lens = _full_lists(w, permute_seed=62)
    got = _run(w, topk_idx=idx, topk_len=lens)
    assert np.max(np.abs(got - _run(w))) < 1e-12


def test_topk_closed_form_on_constant_keys_with_padding_and_duplicates():
    """Constant keys: O = mean of the position tags over the list entries that
    are keys of the row (0 <= j < S_k and j <= i + ctx), counted as listed; -1,
    S_k and causally hidden entries drop out; an empty list gives O = 0."""
    sq, sk = [3, 1, 5], [40, 17, 12]
    w = _constant_key_workload(sq, sk, seed=63)
    g = torch.Generator().manual_seed(64)
    K = 24
    rows, lens = [], []
    for s, i, ctx in token_of_row(w):
        hi = i + ctx
        n = int(torch.randint(0, K + 1, (1,), generator=g))
        ent = torch.randint(-2, sk[s] + 3, (n,), generator=g).to(torch.int32)
        if n >= 2:
            ent[1] = ent[0]                       # one duplicate
        if n >= 3:
            ent[2] = min(hi + 1, sk[s])           # hidden by the causal mask or past S_k
        row = torch.full((K,), -1, dtype=torch.int32)
        row[:n] = ent
        rows.append(row)
        lens.append(n)
    idx, lens_t = torch.stack(rows), torch.tensor(lens, dtype=torch.int32)
    idx[0, :] = -1                                # token 0: an empty list ...
    lens_t[0] = K                                 # ... of K padding entries
    out = _run(w, topk_idx=idx, topk_len=lens_t)
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        ent = idx[tok, :int(lens_t[tok])].numpy().astype(np.int64)
        keep = ent[(ent >= 0) & (ent < sk[s]) & (ent <= i + ctx)]
        for h in range(w.hq):
            if keep.size == 0:
                assert np.all(out[tok, h] == 0)
                continue
            tags = tag_values(keep, h // w.g)
            for k in range(4):
                assert abs(out[tok, h, k] - np.mean(tags[k])) < 1e-12


def test_topk_single_entry_returns_that_value_row_and_window_list_equals_window():
    """One listed key -> O = its V row; the list [i+ctx-W+1 .. i+ctx] equals
    the dense call with window W (same key set)."""
    sq, sk = [4, 2], [30, 9]
    w = _blank(sq, sk, seed=65)
    _random_kv(w, 66)
    W_ = 6
    one, win, lens1, lensw = [], [], [], []
    for s, i, ctx in token_of_row(w):
        j = (7 * i + 3) % (i + ctx + 1)
        r1 = torch.full((W_,), -1, dtype=torch.int32)
        r1[0] = j
        one.append(r1)
        lens1.append(1)
        lo = max(0, i + ctx - W_ + 1)
        rw = torch.full((W_,), -1, dtype=torch.int32)
        rw[:i + ctx - lo + 1] = torch.arange(lo, i + ctx + 1, dtype=torch.int32)
        win.append(rw)
        lensw.append(i + ctx - lo + 1)
    out1 = _run(w, topk_idx=torch.stack(one), topk_len=torch.tensor(lens1, dtype=torch.int32))
    for tok, (s, i, ctx) in enumerate(token_of_row(w)):
        j = (7 * i + 3) % (i + ctx + 1)
        for h in range(w.hq):
            assert decode_tag(out1[tok, h]) == (j, h // w.g)
    outw = _run(w, topk_idx=torch.stack(win), topk_len=torch.tensor(lensw, dtype=torch.int32))
    assert np.max(np.abs(outw - _run(w, window=W_))) < 1e-12


def test_topk_weights_follow_the_list():
    w = _flagged_random(67, sinks=True)
    idx, lens = W.topk_lists(w.seqlens_q, w.seqlens_k, 12, 68, ragged=True, junk=0.3)
    got = _run(w, topk_idx=idx, topk_len=lens)
    for tok in range(0, w.total_q, 5):
        wt, o = oracle.row_weights(w.q, w.k_cache, w.v_cache, w.block_table, w.cu_seqlens_q,
                                   w.seqused_k, w.scale, tok, 2, sinks=w.sinks,
                                   topk_idx=idx, topk_len=lens)
        n = int(lens[tok])
        assert wt.shape == (n + 1,)
        assert abs(wt.sum() - 1.0) < 1e-12
        assert np.max(np.abs(o - got[tok, 2])) < 1e-12


def test_topk_rejects_a_list_longer_than_its_capacity():
    w = _flagged_random(69)
    idx, lens = W.topk_lists(w.seqlens_q, w.seqlens_k, 8, 70)
    lens[1] = 9
    with pytest.raises(oracle.OracleError):
        _run(w, topk_idx=idx, topk_len=lens)

"""Pins for the fp64 oracle, each independent of the oracle's own code.

Every check here would fail for a plausible mistake in the oracle: a dropped
scale, the wrong KV head for a query head (h % Hkv instead of h // g), a wrong
page or slot index, a window that is off by one, a base-2 LSE, a missing
softmax normalisation, or a transposed K/V operand.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from paged_kv_gqa_pa_gb300 import workloads

HERE = os.path.dirname(os.path.abspath(__file__))


def values(a, dtype="f16"):
    """Element values as float64, independently of the oracle: fp16 and fp32
    through numpy, bf16 bit patterns as the upper half of a float32."""
    if dtype == "bf16":
        return (a.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


def _contiguous_kv(case_k, case_v, bt_row, L, ps, dtype="f16"):
    """Gather one sequence's K/V into contiguous [Hkv, L, D] arrays (numpy fancy
    indexing; no code shared with the oracle)."""
    npg = math.ceil(L / ps)
    pages = bt_row[:npg]
    k = values(case_k[pages], dtype)  # [npg, Hkv, ps, D]
    v = values(case_v[pages], dtype)
    Hkv, D = k.shape[1], k.shape[3]
    k = k.transpose(1, 0, 2, 3).reshape(Hkv, npg * ps, D)[:, :L]
    v = v.transpose(1, 0, 2, 3).reshape(Hkv, npg * ps, D)[:, :L]
    return k, v


def _dense_reference(case, window):
    """Textbook attention per sequence on a contiguous copy: fp64
    torch scaled_dot_product_attention with K/V repeated over the head group
    (repeat_interleave: query head h reads KV head h // g), and the LSE from
    torch.logsumexp of the explicit scores."""
    B, Hq, D = case.q.shape
    Hkv = case.k_cache.shape[1]
    g = Hq // Hkv
    out = np.zeros((B, Hq, D))
    lse = np.zeros((B, Hq))
    for b in range(B):
        L = int(case.context_lens[b])
        start = L - window if 0 < window < L else 0
        if L - start == 0:
            lse[b] = -np.inf
            continue
        k, v = _contiguous_kv(case.k_cache, case.v_cache, case.block_tables[b], L,
                              case.page_size, case.dtype)
        k = torch.from_numpy(k[:, start:L]).repeat_interleave(g, dim=0)  # [Hq, n, D]
        v = torch.from_numpy(v[:, start:L]).repeat_interleave(g, dim=0)
        q = torch.from_numpy(values(case.q[b], case.dtype)).unsqueeze(1)  # [Hq, 1, D]
        o = torch.nn.functional.scaled_dot_product_attention(
            q.unsqueeze(0), k.unsqueeze(0), v.unsqueeze(0), scale=case.scale)
        out[b] = o[0, :, 0, :].numpy()
        s = (q @ k.transpose(1, 2))[:, 0, :] * case.scale
        lse[b] = torch.logsumexp(s, dim=-1).numpy()
    return out, lse


SMALL = [
    # B, Hq, Hkv, D, lens, window
    (1, 1, 1, 8, [1], 0),
    (2, 4, 2, 16, [17, 40], 0),
    (3, 6, 2, 32, [5, 33, 64], 0),
    (2, 3, 1, 64, [100, 16], 0),
    (2, 8, 4, 64, [70, 129], 20),
    (1, 4, 4, 128, [48], 48),
    (2, 2, 1, 256, [31, 1], 7),
    (2, 6, 2, 96, [77, 160], 0),
]


@pytest.mark.parametrize("B,Hq,Hkv,D,lens,window", SMALL)
def test_matches_dense_textbook_attention(B, Hq, Hkv, D, lens, window):
    case = workloads.make_case("t", B, Hq, Hkv, D, lens, seed=7 + D + B, window=window,
                               q_std=2.0)
    out, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                             case.context_lens, case.scale, window)
    ref_out, ref_lse = _dense_reference(case, window)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("B,Hq,Hkv,D,lens,window", [SMALL[2], SMALL[4], SMALL[7]])
def test_bf16_inputs_match_dense_textbook_attention(B, Hq, Hkv, D, lens, window):
    case = workloads.make_case("t", B, Hq, Hkv, D, lens, seed=77 + D, window=window,
                               q_std=2.0, dtype="bf16")
    out, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                             case.context_lens, case.scale, window, dtype="bf16")
    ref_out, ref_lse = _dense_reference(case, window)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("B,Hq,Hkv,D,lens,window", [SMALL[2], SMALL[4], SMALL[6]])
def test_fp32_inputs_match_dense_textbook_attention(B, Hq, Hkv, D, lens, window):
    case = workloads.make_case("t", B, Hq, Hkv, D, lens, seed=99 + D, window=window,
                               q_std=2.0, dtype="f32")
    assert case.q.dtype == np.float32
    out, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                             case.context_lens, case.scale, window, dtype="f32")
    ref_out, ref_lse = _dense_reference(case, window)
    np.testing.assert_allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=1e-13, atol=1e-13)


def test_bf16_conversion_is_exact_for_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32)
    with np.errstate(invalid="ignore"):  # signalling-NaN patterns
        ref = (bits << np.uint32(16)).view(np.float32).astype(np.float64)
    got = np.array([oracle.bf16_to_double(int(x)) for x in bits])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_gqa_mapping_is_contiguous_groups():
    # Distinct KV heads: h // g and h % Hkv must give different answers, so this
    # catches the wrong mapping.
    case = workloads.make_case("t", 1, 6, 3, 16, [20], seed=3)
    out, _ = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                           case.context_lens, case.scale)
    ref, _ = _dense_reference(case, 0)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-13)
    # The modulo mapping would disagree with it.
    wrong = case.k_cache[:, [0, 1, 2], :, :]
    alt = workloads.Case(**{**case.__dict__})
    alt.k_cache = np.ascontiguousarray(wrong[:, [0, 0, 1], :, :])
    assert not np.allclose(
        oracle.decode(alt.q, alt.k_cache, case.v_cache, case.block_tables,
                      case.context_lens, case.scale)[0], out)


def _eval_expr(s):
    return eval(s, {"__builtins__": {}}, {"e": math.e, "log": math.log})


def test_closed_form_golden_cases():
    with open(os.path.join(HERE, "golden", "closed_form_cases.json")) as f:
        spec = json.load(f)
    for c in spec["cases"]:
        ps = 16
        Hq, Hkv, D, npg = c["Hq"], c["Hkv"], c["D"], c["num_pages"]
        k = np.full((npg, Hkv, ps, D), np.nan, dtype=np.float16)
        v = np.full((npg, Hkv, ps, D), np.nan, dtype=np.float16)
        for page, rows in c["k_rows"].items():
            for kvh, r in enumerate(rows):
                k[int(page), kvh, :len(r)] = np.array(r, dtype=np.float16)
        for page, rows in c["v_rows"].items():
            for kvh, r in enumerate(rows):
                v[int(page), kvh, :len(r)] = np.array(r, dtype=np.float16)
        q = np.array(c["q"], dtype=np.float16)
        bt = np.array(c["block_table"], dtype=np.int32)
        cl = np.array(c["context_lens"], dtype=np.int32)
        out, lse = oracle.decode(q, k, v, bt, cl, c["scale"], c["window"])
        exp_out = np.vectorize(_eval_expr, otypes=[float])(np.array(c["expect_out"]))
        exp_lse = np.vectorize(_eval_expr, otypes=[float])(np.array(c["expect_lse"]))
        np.testing.assert_allclose(out, exp_out, rtol=1e-14, atol=1e-15, err_msg=c["name"])
        np.testing.assert_allclose(lse, exp_lse, rtol=1e-14, atol=1e-15, err_msg=c["name"])


def test_page_placement_brute_force():
    # Three logical pages placed at every permutation of three physical pages
    # (and the table permuted to match) must give bitwise-identical results.
    base = workloads.make_case("t", 1, 4, 2, 16, [40], seed=11, pool_pages=3)
    logical = base.k_cache[base.block_tables[0, :3]], base.v_cache[base.block_tables[0, :3]]
    results = []
    for perm in itertools.permutations(range(3)):
        k = np.empty_like(base.k_cache)
        v = np.empty_like(base.v_cache)
        for j, phys in enumerate(perm):
            k[phys] = logical[0][j]
            v[phys] = logical[1][j]
        bt = np.array([perm], dtype=np.int32)
        results.append(oracle.decode(base.q, k, v, bt, base.context_lens, base.scale))
    for out, lse in results[1:]:
        assert np.array_equal(out, results[0][0])
        assert np.array_equal(lse, results[0][1])


def test_single_token_returns_v_row_exactly():
    case = workloads.make_case("t", 2, 4, 2, 64, [1, 1], seed=5, q_std=3.0)
    out, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                             case.context_lens, case.scale)
    for b in range(2):
        for h in range(4):
            kvh = h // 2
            page = case.block_tables[b, 0]
            vrow = case.v_cache[page, kvh, 0].astype(np.float64)
            assert np.array_equal(out[b, h], vrow)
            # lse equals the single score, computed exactly with rationals.
            qf = [Fraction(float(x)) for x in case.q[b, h]]
            kf = [Fraction(float(x)) for x in case.k_cache[page, kvh, 0]]
            s = Fraction(case.scale) * sum(a * c for a, c in zip(qf, kf))
            assert lse[b, h] == pytest.approx(float(s), rel=1e-15, abs=1e-15)


def test_zero_query_gives_mean_of_v_and_log_count():
    case = workloads.make_case("t", 3, 2, 1, 32, [1, 37, 80], seed=9, window=0)
    case.q[:] = 0
    for window in (0, 25):
        out, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                 case.context_lens, case.scale, window)
        for b in range(3):
            L = int(case.context_lens[b])
            start = L - window if 0 < window < L else 0
            _, v = _contiguous_kv(case.k_cache, case.v_cache, case.block_tables[b], L, 16)
            mean = v[0, start:L].mean(axis=0)
            np.testing.assert_allclose(out[b, 0], mean, rtol=1e-13, atol=1e-14)
            assert lse[b, 0] == pytest.approx(math.log(L - start), abs=1e-14)


def test_lse_is_logsumexp_of_scores():
    from scipy.special import logsumexp
    case = workloads.make_case("t", 2, 4, 2, 64, [90, 300], seed=13, q_std=3.0)
    _, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                           case.context_lens, case.scale)
    for b in range(2):
        L = int(case.context_lens[b])
        k, _ = _contiguous_kv(case.k_cache, case.v_cache, case.block_tables[b], L, 16)
        for h in range(4):
            s = oracle.scores(case.q, case.k_cache, case.block_tables, case.context_lens,
                              case.scale, 0, b, h)
            # The scores themselves against numpy on the contiguous copy ...
            ref_s = case.scale * (k[h // 2] @ case.q[b, h].astype(np.float64))
            np.testing.assert_allclose(s, ref_s, rtol=1e-13, atol=1e-12)
            # ... and the LSE against scipy's log-sum-exp (natural log).
            assert lse[b, h] == pytest.approx(logsumexp(s), abs=1e-12)


@pytest.mark.parametrize("W", [1, 15, 16, 17, 100])
def test_window_equals_truncated_context(W):
    L = 130
    case = workloads.make_case("t", 1, 2, 1, 16, [L], seed=21)
    out_w, lse_w = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                 case.context_lens, case.scale, W)
    # Copy the last W tokens into fresh pages (different page alignment) and
    # attend all of them with no window.
    k, v = _contiguous_kv(case.k_cache, case.v_cache, case.block_tables[0], L, 16)
    npg = math.ceil(W / 16)
    k2 = np.full((npg, 1, 16, 16), np.nan, dtype=np.float16)
    v2 = np.full_like(k2, np.nan)
    for t in range(W):
        k2[t // 16, 0, t % 16] = k[0, L - W + t].astype(np.float16)
        v2[t // 16, 0, t % 16] = v[0, L - W + t].astype(np.float16)
    bt2 = np.arange(npg, dtype=np.int32)[None, :]
    out_t, lse_t = oracle.decode(case.q, k2, v2, bt2, np.array([W], np.int32), case.scale, 0)
    np.testing.assert_allclose(out_w, out_t, rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(lse_w, lse_t, rtol=1e-14, atol=1e-15)


@pytest.mark.parametrize("W", [0, 130, 131, 1000])
def test_window_at_least_context_is_no_window(W):
    case = workloads.make_case("t", 1, 2, 1, 16, [130], seed=22)
    a = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                      case.context_lens, case.scale, 0)
    b = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                      case.context_lens, case.scale, W)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("S", [16, 48, 64, 200])
def test_partition_then_lse_merge_equals_whole(S):
    """The two-phase algebra (per-partition output + (max, exp-sum), then the
    log-sum-exp merge of the paged_attention_v2_pytorch.py commit note, Phase 2)
    reaches the oracle's one-pass value.  Each partition is run through the
    oracle as its own sequence; the merge is written out here."""
    L = 333
    case = workloads.make_case("t", 1, 4, 2, 32, [L], seed=31, q_std=2.5)
    full_out, full_lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                                       case.context_lens, case.scale)
    k, v = _contiguous_kv(case.k_cache, case.v_cache, case.block_tables[0], L, 16)
    parts = []
    for lo in range(0, L, S):
        hi = min(L, lo + S)
        n = hi - lo
        npg = math.ceil(n / 16)
        k2 = np.full((npg, 2, 16, 32), np.nan, dtype=np.float16)
        v2 = np.full_like(k2, np.nan)
        for t in range(n):
            k2[t // 16, :, t % 16] = k[:, lo + t].astype(np.float16)
            v2[t // 16, :, t % 16] = v[:, lo + t].astype(np.float16)
        bt2 = np.arange(npg, dtype=np.int32)[None, :]
        parts.append(oracle.decode(case.q, k2, v2, bt2, np.array([n], np.int32), case.scale))
    o_p = np.stack([p[0] for p in parts])     # [P, 1, Hq, D], normalised per partition
    lse_p = np.stack([p[1] for p in parts])   # [P, 1, Hq]
    # m_p and l_p are the partition max and exp-sum: lse_p = m_p + log l_p.
    M = lse_p.max(axis=0)
    w = np.exp(lse_p - M)                     # exp(m_p - M) * l_p, up to exp(M) factors
    merged = (w[..., None] * o_p).sum(axis=0) / w.sum(axis=0)[..., None]
    np.testing.assert_allclose(merged, full_out, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(M + np.log(w.sum(axis=0)), full_lse, rtol=1e-13, atol=1e-13)


def test_half_conversion_is_exact_for_every_bit_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32)
    ref = bits.astype(np.uint16).view(np.float16).astype(np.float64)
    got = np.array([oracle.half_to_double(int(x)) for x in bits[::1]])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_empty_context_and_bad_page():
    case = workloads.make_case("t", 2, 2, 1, 16, [0, 20], seed=41)
    out, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                             case.context_lens, case.scale)
    assert np.all(out[0] == 0) and np.all(np.isneginf(lse[0]))
    bad = case.block_tables.copy()
    bad[1, 1] = case.num_pages  # one past the pool
    with pytest.raises(oracle.OracleError):
        oracle.decode(case.q, case.k_cache, case.v_cache, bad, case.context_lens, case.scale)


def test_workload_recipe_shapes():
    # The table is shuffled, pads with -1, and slack pages are NaN.
    c = workloads.workload("tiny_d64")
    assert c.k_cache.shape == (64, 1, 16, 64) and c.block_tables.shape == (1, 16)
    used = set(c.block_tables[0].tolist())
    assert len(used) == 16 and c.block_tables[0].tolist() != list(range(16))
    slack = [p for p in range(64) if p not in used]
    assert np.isnan(c.k_cache[slack].astype(np.float32)).all()
    assert not np.isnan(c.k_cache[sorted(used)].astype(np.float32)).any()
    c3 = workloads.workload("batch8_ragged_d128")
    assert c3.context_lens[0] == 1 and c3.block_tables.shape == (8, 256)
    assert np.any(c3.context_lens % 512 != 0) and c3.context_lens.max() <= 4096


def _rope_complex(x, pos, theta):
    """Rotary embedding written with complex numbers (independent of the
    oracle's pairwise form): the pair (x_i, x_{i+D/2}) is the complex number
    x_i + i x_{i+D/2}, multiplied by exp(i * pos * theta^(-2i/D))."""
    half = x.shape[-1] // 2
    z = x[..., :half] + 1j * x[..., half:]
    freq = theta ** (-2.0 * np.arange(half) / x.shape[-1])
    z = z * np.exp(1j * np.multiply.outer(pos, freq))
    return np.concatenate([z.real, z.imag], axis=-1)


@pytest.mark.parametrize("D,theta", [(64, 10000.0), (128, 500000.0), (256, 10000.0)])
def test_rope_matches_complex_rotation_reference(D, theta):
    lens = [1, 37, 300]
    case = workloads.make_case("r", 3, 4, 2, D, lens, seed=91 + D, window=100)
    out, lse = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                             case.context_lens, case.scale, case.window, rope_theta=theta)
    for b, L in enumerate(lens):
        start = L - case.window if 0 < case.window < L else 0
        k, v = _contiguous_kv(case.k_cache, case.v_cache, case.block_tables[b], L, 16)
        pos = np.arange(L)
        kr = _rope_complex(k, pos, theta)                                 # [Hkv, L, D]
        qr = _rope_complex(case.q[b].astype(np.float64), np.full(4, L - 1.0), theta)
        for h in range(4):
            s = case.scale * (kr[h // 2, start:] @ qr[h])
            w = np.exp(s - s.max())
            np.testing.assert_allclose(out[b, h], (w / w.sum()) @ v[h // 2, start:],
                                       rtol=1e-11, atol=1e-12)
            assert lse[b, h] == pytest.approx(s.max() + np.log(w.sum()), abs=1e-11)


def test_rope_depends_only_on_relative_position():
    """Shifting every position by the same amount leaves the scores unchanged:
    move a context of 40 tokens so that it starts at token 1000 (fresh pages,
    the first 1000 tokens outside a window of 40)."""
    D, theta = 64, 10000.0
    case = workloads.make_case("r", 1, 2, 1, D, [40], seed=95)
    a = oracle.decode(case.q, case.k_cache, case.v_cache, case.block_tables,
                      case.context_lens, case.scale, 0, rope_theta=theta)
    k, v = _contiguous_kv(case.k_cache, case.v_cache, case.block_tables[0], 40, 16)
    L2 = 1040
    npg = math.ceil(L2 / 16)
    k2 = np.zeros((npg, 1, 16, D), dtype=np.float16)
    v2 = np.zeros_like(k2)
    for t in range(40):
        k2[(1000 + t) // 16, 0, (1000 + t) % 16] = k[0, t].astype(np.float16)
        v2[(1000 + t) // 16, 0, (1000 + t) % 16] = v[0, t].astype(np.float16)
    bt2 = np.arange(npg, dtype=np.int32)[None, :]
    b = oracle.decode(case.q, k2, v2, bt2, np.array([L2], np.int32), case.scale, 40,
                      rope_theta=theta)
    np.testing.assert_allclose(b[0], a[0], rtol=1e-9, atol=1e-10)
    np.testing.assert_allclose(b[1], a[1], rtol=1e-10, atol=1e-10)

"""Pins of the fp64 oracle to things other than itself.

Each ``pin_*`` function takes a loaded oracle handle and raises AssertionError when the oracle
disagrees with what the pages or the mathematics fix.  ``test_oracle_pins.py`` runs them on the
real oracle; ``test_oracle_mutants.py`` runs them on builds with one planted mistake each and
requires that every planted mistake fails at least one pin.

What pins what:
  printed worked examples  -> the pages' tables and figures (tests/golden/*.txt, cited there)
  closed forms             -> uniform scores, the causal first row, two keys (logistic form),
                              constant values, scale 0
  library special case     -> scipy.special.softmax / logsumexp for the row softmax
  exact brute force        -> 40-digit decimal arithmetic by the textbook formula (highprec.py)
  invariants               -> rows sum to 1, shift invariance, key permutation invariance,
                              block-size independence, the two-worker merge law
"""
from __future__ import annotations

import math

import numpy as np
import torch

import golden_io
import highprec
from online_softmax_tiled_attn_gb300 import inputs


def _bits(values, shape):
    t = torch.tensor(values, dtype=torch.float32).reshape(shape).to(torch.bfloat16)
    return inputs.bf16_bits(t)


def _bf16_float(t):
    return t.to(torch.float32).numpy().astype(np.float64)


def _row_attention(orc, s, v):
    """Attention of one query whose scores are s (given exactly) with values v, via the
    three-pass oracle: d=1 keys k_j = s_j, q = 1, scale = 1 needs bf16-exact scores, so use
    the softmax oracle for the weights instead when s is arbitrary."""
    y, lse = orc.softmax_rows(np.asarray(s, dtype=np.float32)[None, :])
    return y[0] @ np.asarray(v, dtype=np.float64), y[0], lse[0]


# ----------------------------------------------------------------------------------------------
# printed worked examples
# ----------------------------------------------------------------------------------------------

def pin_four_scores_all_at_once(orc):
    g = golden_io.load("four_scores_kbwen.txt")
    s, v = g["scores"], g["values"]
    Q = _bits([1.0], (1, 1, 1, 1))
    K = _bits(s, (1, 1, 4, 1))
    V = _bits(v, (1, 1, 4, 1))
    # the query is repeated as 4 rows so every row sees all four keys (non-causal)
    Q4 = np.repeat(Q, 4, axis=2)
    O, L = orc.attention(Q4, K, V, 1.0, False)
    for i in range(4):
        assert abs(O[0, 0, i, 0] - g["output_8dp"][0]) < 5e-9, O[0, 0, i, 0]
    assert round(O[0, 0, 0, 0], 4) == g["output_4dp"][0]
    m = max(s)
    lsum = math.exp(L[0, 0, 0] - m)
    assert round(lsum, 4) == g["sum_4dp"][0], lsum
    assert round(O[0, 0, 0, 0] * lsum, 4) == g["weighted_sum_4dp"][0]
    y, _ = orc.softmax_rows(np.array([s], dtype=np.float32))
    assert [round(w, 4) for w in (y[0] * lsum)] == g["weights_4dp"]


def pin_four_scores_two_blocks(orc):
    g = golden_io.load("four_scores_kbwen.txt")
    st = orc.online_state(g["scores"], g["values"], block=2, trace=True)
    assert list(st["trace_m"]) == [g["block1_max"][0], max(g["scores"])]
    l1, a1 = st["trace_l"][0], st["trace_acc"][0, 0]
    assert round(l1, 4) == g["block1_sum_4dp"][0]
    assert round(a1, 4) == g["block1_weighted_sum_4dp"][0]
    assert round(a1 / l1, 2) == g["block1_output_2dp"][0]
    alpha = st["trace_alpha"][1]
    assert round(alpha, 4) == g["rescale_factor_4dp"][0]
    assert round(l1 * alpha, 4) == g["carried_sum_after_rescale_4dp"][0]
    assert round(a1 * alpha, 4) == g["carried_weighted_sum_after_rescale_4dp"][0]
    assert round(st["trace_psum"][1], 4) == g["block2_sum_4dp"][0]
    assert round(st["trace_acc"][1, 0] - a1 * alpha, 4) == g["block2_weighted_sum_4dp"][0]
    assert round(st["l"], 4) == g["sum_4dp"][0]
    assert round(st["acc"][0], 4) == g["weighted_sum_4dp"][0]
    assert abs(st["acc"][0] / st["l"] - g["output_8dp"][0]) < 5e-9


def pin_four_scores_random_blocks(orc):
    """The page's random check: 1000 scores N(0, sd 4), 8-wide values, blocks of 64."""
    g = golden_io.load("four_scores_kbwen.txt")
    rng = np.random.default_rng(0)
    s = rng.normal(0, 4, size=1000)
    v = rng.normal(size=(1000, 8))
    st = orc.online_state(s, v, block=64)
    streamed = st["acc"] / st["l"]
    y, _ = orc.softmax_rows(s.astype(np.float32)[None, :])
    # compare against the three-pass weights on the same (fp32-rounded) scores
    st32 = orc.online_state(s.astype(np.float32).astype(np.float64), v, block=64)
    diff = np.abs(st32["acc"] / st32["l"] - y[0] @ v).max()
    assert diff < 100 * g["random_max_abs_diff"][0], diff
    assert np.all(np.isfinite(streamed))


def pin_counter_example(orc):
    g = golden_io.load("counter_example_dubiel.txt")
    # scores 0, 0, ln3, ln3 enter as keys 0, 0, 1, 1 with q = 1 and scale = ln 3 (fp64)
    Q = _bits([1.0], (1, 1, 1, 1))
    K = _bits([0.0, 0.0, 1.0, 1.0], (1, 1, 4, 1))
    V = _bits(g["values"], (1, 1, 4, 1))
    O, L = orc.attention(np.repeat(Q, 4, axis=2), K, V, math.log(3.0), False)
    assert abs(O[0, 0, 0, 0] - g["result"][0]) < 1e-15, O[0, 0, 0, 0]
    assert abs(L[0, 0, 0] - math.log(8.0)) < 1e-15  # 1 + 1 + 3 + 3 = 8
    # block results on their own are 0 and 1; their plain mean is the wrong 0.5
    b1 = orc.online_state(g["scores"][:2], g["values"][:2], block=2)
    b2 = orc.online_state(g["scores"][2:], g["values"][2:], block=2)
    assert [b1["acc"][0] / b1["l"], b2["acc"][0] / b2["l"]] == g["block_results"]
    st = orc.online_state(g["scores"], g["values"], block=2)
    assert abs(st["acc"][0] / st["l"] - g["result"][0]) < 1e-15
    assert abs(st["acc"][0] / st["l"] - g["wrong_block_mean"][0]) > 0.2
    w = np.exp(np.array(g["scores"]) - min(g["scores"]))
    assert np.allclose(w, g["weight_proportions"], rtol=1e-15)


def pin_five_scores_table(orc):
    g = golden_io.load("five_scores_spicyshark.txt")
    x, v = g["scores"], g["values"]
    st = orc.online_state(x, v, block=1, trace=True)
    assert list(st["trace_m"]) == g["m"]
    assert [round(a, 5) for a in st["trace_alpha"]] == g["alpha_5dp"]
    assert [round(p, 5) for p in st["trace_psum"]] == g["new_term_5dp"]
    assert [round(l, 4) for l in st["trace_l"]] == g["l_4dp"]
    acc = st["trace_acc"][:, 0]
    assert [round(a, 4) for a in acc] == g["acc_full_precision_4dp"]
    assert np.abs(acc - np.array(g["acc_by_hand_4dp"])).max() < g["by_hand_vs_full_max_diff"][0]
    assert [round(a / l, 2) for a, l in zip(acc, st["trace_l"])] == g["output_2dp"]
    y, lse = orc.softmax_rows(np.array([x], dtype=np.float32))
    assert [round(p, 4) for p in y[0]] == g["probabilities_4dp"]
    l_final = math.exp(lse[0] - 5.0)
    assert [round(p * l_final, 5) for p in y[0]] == g["exp_x_minus_5_5dp"]
    hand = np.array(g["probabilities_4dp"]) @ np.array(v)
    assert round(hand, 3) == g["textbook_weighted_sum_3dp"][0]
    st2 = orc.online_state(x, v, block=2, trace=True)
    assert [round(l, 4) for l in st2["trace_l"]] == g["blocks_of_two_l_4dp"]
    # the three-pass attention of the same query equals the streamed answer
    Q = _bits([1.0] * 5, (1, 1, 5, 1))
    O, _ = orc.attention(Q, _bits(x, (1, 1, 5, 1)), _bits(v, (1, 1, 5, 1)), 1.0, False)
    assert abs(O[0, 0, 4, 0] - st["acc"][0] / st["l"]) < 1e-12
    assert round(O[0, 0, 4, 0], 2) == g["output_2dp"][-1]


def pin_overflow_row(orc):
    g = golden_io.load("overflow_and_masking_spicyshark.txt")
    row = np.array([g["fp32_row"]], dtype=np.float32)
    with np.errstate(over="ignore"):
        assert np.isfinite(np.exp(np.float32(g["fp32_exp_finite_at"][0])))
        assert np.isinf(np.exp(np.float32(g["fp32_exp_overflows_at"][0])))
    y, lse = orc.softmax_rows(row)
    t = np.exp(np.array(g["fp32_row_softmax_equals_softmax_of"]))
    want = t / t.sum()
    assert np.abs(y[0] - want).max() < g["fp32_row_atol"][0]
    assert np.abs(y[0] - want).max() < 1e-15
    assert abs(lse[0] - (1002.0 + math.log(t.sum()))) < 1e-12


def pin_masked_prefix(orc):
    g = golden_io.load("overflow_and_masking_spicyshark.txt")
    blocks = g["masked_stats_blocks"]
    s = blocks[0] + blocks[1]
    st = orc.online_state(s, np.zeros(len(s)), block=len(blocks[0]))
    assert st["m"] == g["masked_stats_m"][0]
    assert abs(st["l"] - (math.exp(-1.0) + 1.0)) < 1e-15
    # both sides get the same fp32-exact scores (the softmax oracle reads fp32 rows)
    sc = np.array(g["masked_attention_scores"], dtype=np.float32).astype(np.float64)
    V = np.random.default_rng(5).standard_normal((len(sc), 3))
    st = orc.online_state(sc, V, block=int(g["masked_attention_block"][0]))
    assert st["m"] == 2.0 and math.isfinite(st["l"]) and np.all(np.isfinite(st["acc"]))
    out, y, _ = _row_attention(orc, sc, V)
    assert y[0] == 0.0 and y[1] == 0.0
    assert np.abs(st["acc"] / st["l"] - out).max() < 1e-14
    # a row with no finite score: the softmax is all zeros and the log-sum-exp is -inf
    yz, lz = orc.softmax_rows(np.full((1, 4), -np.inf, dtype=np.float32))
    assert np.all(yz == 0.0) and lz[0] == -np.inf


# ----------------------------------------------------------------------------------------------
# library special case and exact brute force
# ----------------------------------------------------------------------------------------------

def pin_softmax_matches_scipy(orc):
    from scipy.special import logsumexp, softmax

    x = inputs.softmax_inputs(7, 53, seed=11, std=9.0, spike=100.0).numpy()
    y, lse = orc.softmax_rows(x)
    xd = x.astype(np.float64)
    assert np.abs(y - softmax(xd, axis=1)).max() < 1e-15
    assert np.abs(lse - logsumexp(xd, axis=1)).max() < 1e-12
    assert np.abs(y.sum(axis=1) - 1.0).max() < 1e-14


def pin_attention_decimal_bruteforce(orc):
    cases = [
        (1, 1, 5, 3, 0.37, False),
        (1, 2, 7, 4, 0.61, True),
        (2, 1, 9, 2, 1.3, False),
        (1, 1, 6, 5, 0.5, True),
    ]
    for seed, (B, H, N, d, scale, causal) in enumerate(cases):
        q, k, v = inputs.attn_inputs(B, H, N, d, seed=77 + seed, qk_std=1.5)
        O, L = orc.attention(q, k, v, scale, causal)
        Od, Ld = highprec.attention_decimal(_bf16_float(q).tolist(), _bf16_float(k).tolist(),
                                            _bf16_float(v).tolist(), scale, causal)
        assert np.abs(O - np.array(Od)).max() < 1e-13, (B, H, N, d, causal)
        assert np.abs(L - np.array(Ld)).max() < 1e-13, (B, H, N, d, causal)


def pin_attention_qk_decimal_bruteforce(orc):
    """Nq queries against Nk keys (the split-key path's definition), causal and not."""
    cases = [(1, 2, 1, 9, 4, 0.45, True), (1, 1, 3, 8, 3, 0.8, True), (2, 1, 4, 7, 2, 1.1, False),
             (1, 1, 5, 5, 3, 0.6, True)]
    for seed, (B, H, Nq, Nk, d, scale, causal) in enumerate(cases):
        q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=91 + seed, qk_std=1.5)
        _, k, v = inputs.attn_inputs(B, H, Nk, d, seed=191 + seed, qk_std=1.5)
        O, L = orc.attention_qk(q, k, v, scale, causal)
        Od, Ld = highprec.attention_decimal(_bf16_float(q).tolist(), _bf16_float(k).tolist(),
                                            _bf16_float(v).tolist(), scale, causal)
        assert np.abs(O - np.array(Od)).max() < 1e-13, (B, H, Nq, Nk, causal)
        assert np.abs(L - np.array(Ld)).max() < 1e-13, (B, H, Nq, Nk, causal)


def pin_attention_qk_square_is_attention(orc):
    q, k, v = inputs.attn_inputs(1, 2, 17, 8, seed=23)
    for causal in (False, True):
        O, L = orc.attention(q, k, v, 0.3, causal)
        O2, L2 = orc.attention_qk(q, k, v, 0.3, causal)
        assert np.array_equal(O, O2) and np.array_equal(L, L2)


def pin_split_keys_merge_to_full(orc):
    """Attention over disjoint key ranges, merged by the two-worker merge, equals attention over
    all keys (the Flash-Decoding combination).  A range state (O_s, LSE_s) is the state
    (m = LSE_s, l = 1, acc = O_s): same acc / l and same m + ln l."""
    B, H, Nq, Nk, d = 1, 1, 3, 50, 4
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=31)
    _, k, v = inputs.attn_inputs(B, H, Nk, d, seed=32)
    O, L = orc.attention_qk(q, k, v, 0.5, False)
    for cuts in ((0, 17, 50), (0, 1, 2, 49, 50), (0, 25, 25, 50)):
        for i in range(Nq):
            st = dict(m=-math.inf, l=0.0, acc=np.zeros(d))
            for a, b in zip(cuts[:-1], cuts[1:]):
                if a == b:
                    part = dict(m=-math.inf, l=0.0, acc=np.zeros(d))  # an empty range
                else:
                    Os, Ls = orc.attention_qk(q[:, :, i:i + 1], k[:, :, a:b], v[:, :, a:b], 0.5,
                                              False)
                    part = dict(m=float(Ls[0, 0, 0]), l=1.0, acc=Os[0, 0, 0])
                st = orc.merge(st, part)
            assert np.abs(st["acc"] / st["l"] - O[0, 0, i]).max() < 1e-13
            assert abs(st["m"] + math.log(st["l"]) - L[0, 0, i]) < 1e-12


def pin_gqa_key_lengths_decimal_bruteforce(orc):
    """Grouped heads and per-sequence key lengths, against the 40-digit textbook formula.  A
    sequence with no key (length 0) must give O = 0 and LSE = -inf (the empty state)."""
    cases = [(2, 4, 2, 3, 6, 3, 0.7, False, [6, 2]), (2, 4, 1, 4, 5, 2, 0.9, True, [5, 3]),
             (1, 6, 3, 2, 7, 3, 0.5, True, [4]), (2, 2, 2, 2, 4, 2, 1.2, False, [0, 3])]
    for seed, (B, H, H_kv, Nq, Nk, d, scale, causal, lens) in enumerate(cases):
        q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=301 + seed, qk_std=1.5)
        _, k, v = inputs.attn_inputs(B, H_kv, Nk, d, seed=401 + seed, qk_std=1.5)
        O, L = orc.attention_gqa(q, k, v, scale, causal, kv_lens=np.array(lens, np.int32))
        Od, Ld = highprec.attention_decimal_gqa(_bf16_float(q).tolist(), _bf16_float(k).tolist(),
                                                _bf16_float(v).tolist(), scale, causal, lens)
        assert np.abs(O - np.array(Od)).max() < 1e-13, (B, H, H_kv, causal, lens)
        Ld = np.array(Ld)
        assert np.array_equal(np.isinf(L), np.isinf(Ld)), (B, H, H_kv, causal, lens)
        fin = np.isfinite(Ld)
        assert np.abs(L[fin] - Ld[fin]).max() < 1e-13, (B, H, H_kv, causal, lens)


def pin_key_padding_ignores_what_lies_beyond(orc):
    """Keys at or past a sequence's length take no part: whatever sits there (here, huge keys
    that would dominate every softmax and huge values) cannot change O or LSE."""
    B, H, Nq, Nk, d = 2, 2, 4, 9, 3
    q, k, v = inputs.attn_inputs(B, H, Nq, d, seed=61)
    _, k, v = inputs.attn_inputs(B, H, Nk, d, seed=62)
    lens = np.array([5, 7], np.int32)
    O, L = orc.attention_gqa(q, k, v, 0.8, False, kv_lens=lens)
    k2, v2 = k.clone(), v.clone()
    for b in range(B):
        k2[b, :, lens[b]:] = 30.0
        v2[b, :, lens[b]:] = -1000.0
    O2, L2 = orc.attention_gqa(q, k2, v2, 0.8, False, kv_lens=lens)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    # ... and a length of Nk is the same as no lengths at all
    O3, L3 = orc.attention_gqa(q, k, v, 0.8, True, kv_lens=np.array([Nk, Nk], np.int32))
    O4, L4 = orc.attention_qk(q, k, v, 0.8, True)
    assert np.array_equal(O3, O4) and np.array_equal(L3, L4)


def pin_gqa_is_attention_with_shared_heads(orc):
    """Grouped heads are the plain attention of each query head with its group's key/value
    head: query heads 2g and 2g+1 of H = 4 read key/value head g of H_kv = 2."""
    B, H, H_kv, N, d = 1, 4, 2, 6, 3
    q, _, _ = inputs.attn_inputs(B, H, N, d, seed=71)
    _, k, v = inputs.attn_inputs(B, H_kv, N, d, seed=72)
    O, L = orc.attention_gqa(q, k, v, 0.6, True)
    for h in range(H):
        g = h // 2
        Oh, Lh = orc.attention(q[:, h:h + 1], k[:, g:g + 1], v[:, g:g + 1], 0.6, True)
        assert np.array_equal(O[:, h:h + 1], Oh) and np.array_equal(L[:, h:h + 1], Lh)


def pin_mask_decimal_bruteforce(orc):
    """An explicit mask (random entries, a fully masked query row, a key masked for every query;
    alone and with the causal mask, key lengths and grouped heads), against the 40-digit
    textbook formula.  A row with no allowed key gives O = 0 and LSE = -inf."""
    cases = [(2, 2, 2, 5, 7, 3, 0.8, False, None, 0.6), (1, 4, 2, 6, 6, 2, 1.1, True, [5], 0.7),
             (2, 2, 1, 4, 9, 3, 0.5, False, [9, 4], 0.3), (1, 1, 1, 7, 7, 4, 0.9, True, None, 1.0)]
    for seed, (B, H, H_kv, Nq, Nk, d, scale, causal, lens, dens) in enumerate(cases):
        q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=901 + seed, qk_std=1.5)
        _, k, v = inputs.attn_inputs(B, H_kv, Nk, d, seed=911 + seed, qk_std=1.5)
        m = inputs.random_mask(B, H, Nq, Nk, dens, seed=921 + seed, full_rows=1, full_keys=1)
        kl = None if lens is None else np.array(lens, np.int32)
        O, L = orc.attention_gqa(q, k, v, scale, causal, kv_lens=kl, mask=m)
        Od, Ld = highprec.attention_decimal_gqa(_bf16_float(q).tolist(), _bf16_float(k).tolist(),
                                                _bf16_float(v).tolist(), scale, causal, lens,
                                                mask=m.astype(bool).tolist())
        what = (B, H, H_kv, causal, lens, dens)
        assert np.abs(O - np.array(Od)).max() < 1e-13, what
        Ld = np.array(Ld)
        assert np.isinf(Ld).any(), what  # the fully masked rows
        assert np.array_equal(np.isinf(L), np.isinf(Ld)), what
        fin = np.isfinite(Ld)
        assert np.abs(L[fin] - Ld[fin]).max() < 1e-13, what


def pin_mask_patterns(orc):
    """Masks that state another rule give that rule's result bit for bit: all ones = no mask,
    the lower triangle = the causal flag, a prefix of each sequence = its key length; a mask
    given once for all heads = the same mask repeated."""
    B, H, N, d = 2, 3, 11, 4
    q, k, v = inputs.attn_inputs(B, H, N, d, seed=931)
    O0, L0 = orc.attention(q, k, v, 0.7, False)
    O1, L1 = orc.attention_gqa(q, k, v, 0.7, False, mask=np.ones((1, 1, N, N), np.uint8))
    assert np.array_equal(O0, O1) and np.array_equal(L0, L1)
    Oc, Lc = orc.attention(q, k, v, 0.7, True)
    Om, Lm = orc.attention_gqa(q, k, v, 0.7, False, mask=np.tril(np.ones((N, N), np.uint8))[None, None])
    assert np.array_equal(Oc, Om) and np.array_equal(Lc, Lm)
    lens = [7, 3]
    pref = np.zeros((B, 1, N, N), np.uint8)
    for b, n in enumerate(lens):
        pref[b, :, :, :n] = 1
    Ok, Lk = orc.attention_gqa(q, k, v, 0.7, False, kv_lens=np.array(lens, np.int32))
    Op, Lp = orc.attention_gqa(q, k, v, 0.7, False, mask=pref)
    assert np.array_equal(Ok, Op) and np.array_equal(Lk, Lp)
    m = inputs.random_mask(1, 1, N, N, 0.5, seed=932)
    Ob, Lb = orc.attention_gqa(q, k, v, 0.7, False, mask=m)
    Or, Lr = orc.attention_gqa(q, k, v, 0.7, False, mask=np.broadcast_to(m, (B, H, N, N)))
    assert np.array_equal(Ob, Or) and np.array_equal(Lb, Lr)


def pin_mask_ignores_masked_keys(orc):
    """A key masked for every query takes no part: huge keys and values planted there change
    nothing."""
    B, H, N, d = 1, 2, 8, 3
    q, k, v = inputs.attn_inputs(B, H, N, d, seed=941)
    m = inputs.random_mask(B, H, N, N, 0.8, seed=942)
    m[:, :, :, 5] = 0
    O, L = orc.attention_gqa(q, k, v, 0.9, False, mask=m)
    k2, v2 = k.clone(), v.clone()
    k2[:, :, 5] = 50.0
    v2[:, :, 5] = -1000.0
    O2, L2 = orc.attention_gqa(q, k2, v2, 0.9, False, mask=m)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)


def pin_closed_form_single_valid_key(orc):
    """A sequence of length 1: every query sees key 0 alone, so O = V_0 and LSE = s_0."""
    B, H, Nq, Nk, d = 1, 2, 3, 5, 4
    q, _, _ = inputs.attn_inputs(B, H, Nq, d, seed=81)
    _, k, v = inputs.attn_inputs(B, H, Nk, d, seed=82)
    O, L = orc.attention_gqa(q, k, v, 0.4, False, kv_lens=np.array([1], np.int32))
    qf, kf, vf = _bf16_float(q), _bf16_float(k), _bf16_float(v)
    for h in range(H):
        for i in range(Nq):
            assert np.abs(O[0, h, i] - vf[0, h, 0]).max() < 1e-15
            s0 = 0.4 * float(np.dot(qf[0, h, i].astype(np.float64), kf[0, h, 0]))
            assert abs(L[0, h, i] - s0) < 1e-12


def pin_softmax_topk_brute_force(orc):
    """Top-k against Python's own sort of (value descending, column ascending) and the shares
    against scipy's softmax; rows with repeated values, -inf entries and the overflow row."""
    from scipy.special import softmax

    g = np.random.default_rng(5)
    x = g.integers(-3, 4, size=(40, 23)).astype(np.float32)  # many ties
    x[3, :20] = -np.inf
    x[7] = np.float32([1000, 1001, 1002] * 7 + [1000, 1000])
    x[9] = g.standard_normal(23).astype(np.float32) * 30
    for k in (1, 2, 5, 23):
        vals, idx, lse = orc.softmax_topk(x, k)
        for r in range(x.shape[0]):
            want = sorted(range(23), key=lambda j: (-float(x[r, j]), j))[:k]
            assert list(idx[r]) == want, (r, k)
            y = softmax(x[r].astype(np.float64))
            assert np.abs(vals[r] - y[want]).max() < 1e-15, (r, k)


def pin_softmax_topk_full_is_sorted_softmax(orc):
    """k = cols: every share once, in order, summing to 1; k = 1 is the arg-max."""
    x = inputs.softmax_inputs(6, 50, seed=17)
    vals, idx, lse = orc.softmax_topk(x.numpy(), 50)
    assert np.all(np.diff(vals, axis=1) <= 0)
    assert np.abs(vals.sum(axis=1) - 1.0).max() < 1e-14
    assert all(sorted(r) == list(range(50)) for r in idx.tolist())
    v1, i1, _ = orc.softmax_topk(x.numpy(), 1)
    assert np.array_equal(i1[:, 0], np.argmax(x.numpy(), axis=1))
    y, l2 = orc.softmax_rows(x.numpy())
    assert np.array_equal(lse, l2) and np.array_equal(v1[:, 0], y.max(axis=1))


def _forward_fp64(q, k, v, scale, causal):
    """O of the definition in plain numpy fp64 (an implementation independent of the oracle),
    [H, N, d] inputs."""
    s = scale * np.einsum("hid,hjd->hij", q, k)
    if causal:
        n = s.shape[-1]
        s = np.where(np.tril(np.ones((n, n), bool)), s, -np.inf)
    p = np.exp(s - s.max(axis=-1, keepdims=True))
    p /= p.sum(axis=-1, keepdims=True)
    return np.einsum("hij,hjd->hid", p, v)


def pin_attention_bwd_finite_differences(orc):
    """The gradients against central differences of L = sum(dO * O) through the definition."""
    for causal in (False, True):
        q, k, v = inputs.attn_inputs(1, 2, 5, 3, seed=501 + causal)
        g, _, _ = inputs.attn_inputs(1, 2, 5, 3, seed=601 + causal)
        dQ, dK, dV = orc.attention_bwd(q, k, v, g, 0.7, causal)
        qf, kf, vf, gf = (_bf16_float(t)[0].astype(np.float64) for t in (q, k, v, g))

        def loss(qq, kk, vv):
            return float((gf * _forward_fp64(qq, kk, vv, 0.7, causal)).sum())

        eps = 1e-5
        for which, grad in ((0, dQ), (1, dK), (2, dV)):
            args = [qf, kf, vf]
            num = np.zeros_like(qf)
            for idx in np.ndindex(qf.shape):
                plus = [a.copy() for a in args]
                minus = [a.copy() for a in args]
                plus[which][idx] += eps
                minus[which][idx] -= eps
                num[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert np.abs(grad[0] - num).max() < 1e-7 * max(1.0, np.abs(num).max()), (which, causal)


def pin_attention_bwd_key_gradients_sum_to_zero(orc):
    """Each row of dS sums to zero (the softmax's shares sum to one), so the key gradients of a
    head sum to the zero vector: sum_j dK_j = scale sum_i Q_i sum_j dS_ij = 0."""
    q, k, v = inputs.attn_inputs(2, 2, 33, 8, seed=701)
    g, _, _ = inputs.attn_inputs(2, 2, 33, 8, seed=702)
    for causal in (False, True):
        _, dK, _ = orc.attention_bwd(q, k, v, g, 0.4, causal)
        assert np.abs(dK.sum(axis=2)).max() < 1e-12, causal


def pin_attention_bwd_uniform_scores(orc):
    """Q = 0: every allowed key gets the same share, so dV_j = sum over the queries that see
    key j of dO_i / (their number of keys): the mean of dO (non-causal), sum_{i>=j} dO_i/(i+1)
    (causal)."""
    N, d = 6, 4
    _, k, v = inputs.attn_inputs(1, 1, N, d, seed=801)
    g, _, _ = inputs.attn_inputs(1, 1, N, d, seed=802)
    q = k.clone()
    q.zero_()
    gf = _bf16_float(g)[0, 0].astype(np.float64)
    _, _, dV = orc.attention_bwd(q, k, v, g, 0.5, False)
    assert np.abs(dV[0, 0] - gf.mean(axis=0)).max() < 1e-14
    _, _, dV = orc.attention_bwd(q, k, v, g, 0.5, True)
    want = np.array([sum(gf[i] / (i + 1) for i in range(j, N)) for j in range(N)])
    assert np.abs(dV[0, 0] - want).max() < 1e-14


def _forward_fp64_gqa(q, k, v, scale, causal, lens):
    """O of the definition in plain numpy fp64 with grouped key/value heads and key lengths:
    q [B, H, N, d], k, v [B, H_kv, N, d]; key j allowed for query i of sequence b when
    j < lens[b] (and j <= i when causal); a row with no allowed key gives 0."""
    B, H, N, _ = q.shape
    group = H // k.shape[1]
    kr = np.repeat(k, group, axis=1)
    vr = np.repeat(v, group, axis=1)
    s = scale * np.einsum("bhid,bhjd->bhij", q, kr)
    allowed = np.ones((B, 1, N, N), bool)
    allowed &= (np.arange(N)[None, None, None, :] < np.asarray(lens)[:, None, None, None])
    if causal:
        allowed &= np.tril(np.ones((N, N), bool))[None, None]
    s = np.where(allowed, s, -np.inf)
    mx = s.max(axis=-1, keepdims=True)
    p = np.where(allowed, np.exp(s - np.where(np.isfinite(mx), mx, 0.0)), 0.0)
    den = p.sum(axis=-1, keepdims=True)
    p = np.divide(p, den, out=np.zeros_like(p), where=den > 0)
    return np.einsum("bhij,bhjd->bhid", p, vr)


def pin_attention_bwd_grouped_heads_finite_differences(orc):
    """Grouped key/value heads and key lengths: the gradients against central differences of
    L = sum(dO * O) through an independent forward (a sequence with fewer keys than N)."""
    B, H, Hkv, N, d, lens = 2, 4, 2, 5, 3, [5, 3]
    for causal in (False, True):
        q, _, _ = inputs.attn_inputs(B, H, N, d, seed=511 + causal)
        _, k, v = inputs.attn_inputs(B, Hkv, N, d, seed=521 + causal)
        g, _, _ = inputs.attn_inputs(B, H, N, d, seed=531 + causal)
        dQ, dK, dV = orc.attention_bwd(q, k, v, g, 0.6, causal,
                                       kv_lens=np.array(lens, np.int32))
        qf, kf, vf, gf = (_bf16_float(t).astype(np.float64) for t in (q, k, v, g))

        def loss(qq, kk, vv):
            return float((gf * _forward_fp64_gqa(qq, kk, vv, 0.6, causal, lens)).sum())

        eps = 1e-5
        for which, grad in ((0, dQ), (1, dK), (2, dV)):
            args = [qf, kf, vf]
            num = np.zeros_like(args[which])
            for idx in np.ndindex(args[which].shape):
                plus = [a.copy() for a in args]
                minus = [a.copy() for a in args]
                plus[which][idx] += eps
                minus[which][idx] -= eps
                num[idx] = (loss(*plus) - loss(*minus)) / (2 * eps)
            assert np.abs(grad - num).max() < 1e-7 * max(1.0, np.abs(num).max()), (which, causal)


def pin_attention_bwd_grouped_heads_repeat_law(orc):
    """Grouped heads are the same attention with each key/value head repeated for its query
    heads; a shared head's gradients are the sums of the repeated copies' gradients (the chain
    rule for a shared parameter), and dQ is unchanged."""
    B, H, N, d = 2, 6, 9, 5
    for Hkv in (1, 2, 3):
        q, _, _ = inputs.attn_inputs(B, H, N, d, seed=541 + Hkv)
        _, k, v = inputs.attn_inputs(B, Hkv, N, d, seed=551 + Hkv)
        g, _, _ = inputs.attn_inputs(B, H, N, d, seed=561 + Hkv)
        for causal in (False, True):
            dQ, dK, dV = orc.attention_bwd(q, k, v, g, 0.45, causal)
            kr = k.repeat_interleave(H // Hkv, dim=1)
            vr = v.repeat_interleave(H // Hkv, dim=1)
            dQr, dKr, dVr = orc.attention_bwd(q, kr, vr, g, 0.45, causal)
            assert np.abs(dQ - dQr).max() < 1e-13
            sumK = dKr.reshape(B, Hkv, H // Hkv, N, d).sum(axis=2)
            sumV = dVr.reshape(B, Hkv, H // Hkv, N, d).sum(axis=2)
            assert np.abs(dK - sumK).max() < 1e-12 and np.abs(dV - sumV).max() < 1e-12


def pin_attention_bwd_key_lengths(orc):
    """Keys at or past a sequence's length take no part: their gradients are exactly 0, and
    values planted there change no gradient; a sequence of length 0 has all gradients 0."""
    B, H, Hkv, N, d = 3, 4, 2, 11, 6
    lens = np.array([11, 4, 0], np.int32)
    q, _, _ = inputs.attn_inputs(B, H, N, d, seed=571)
    _, k, v = inputs.attn_inputs(B, Hkv, N, d, seed=572)
    g, _, _ = inputs.attn_inputs(B, H, N, d, seed=573)
    for causal in (False, True):
        dQ, dK, dV = orc.attention_bwd(q, k, v, g, 0.5, causal, kv_lens=lens)
        for b in range(B):
            assert np.all(dK[b, :, lens[b]:] == 0) and np.all(dV[b, :, lens[b]:] == 0)
        assert np.all(dQ[2] == 0) and np.all(dK[2] == 0) and np.all(dV[2] == 0)
        k2, v2 = k.clone(), v.clone()
        k2[1, :, 4:] = 50.0
        v2[1, :, 4:] = -30.0
        dQ2, dK2, dV2 = orc.attention_bwd(q, k2, v2, g, 0.5, causal, kv_lens=lens)
        assert np.array_equal(dQ, dQ2) and np.array_equal(dK, dK2) and np.array_equal(dV, dV2)


# ----------------------------------------------------------------------------------------------
# closed forms
# ----------------------------------------------------------------------------------------------

def pin_closed_form_uniform_scores(orc):
    """All keys equal: every allowed key gets the same weight, so O is the mean of the
    allowed value rows and LSE = s + ln(#allowed)."""
    B, H, N, d = 1, 2, 11, 4
    q, _, v = inputs.attn_inputs(B, H, N, d, seed=5)
    krow = torch.tensor([0.5, -1.0, 0.25, 2.0]).to(torch.bfloat16)
    k = krow.expand(B, H, N, d).contiguous()
    qf, kf, vf = _bf16_float(q), _bf16_float(k), _bf16_float(v)
    for causal in (False, True):
        O, L = orc.attention(q, k, v, 0.3, causal)
        for h in range(H):
            for i in range(N):
                n_allowed = i + 1 if causal else N
                want = vf[0, h, :n_allowed].mean(axis=0)
                s = 0.3 * float(qf[0, h, i] @ kf[0, h, 0])
                assert np.abs(O[0, h, i] - want).max() < 1e-14
                assert abs(L[0, h, i] - (s + math.log(n_allowed))) < 1e-13


def pin_closed_form_last_query_sees_all_keys(orc):
    """With the queries at the end of the key positions, the last query is not masked at all:
    causal and non-causal agree for it, and a single causal query equals full attention."""
    q, _, _ = inputs.attn_inputs(1, 2, 3, 8, seed=41)
    _, k, v = inputs.attn_inputs(1, 2, 12, 8, seed=42)
    Oc, Lc = orc.attention_qk(q, k, v, 0.4, True)
    On, Ln = orc.attention_qk(q, k, v, 0.4, False)
    assert np.array_equal(Oc[:, :, -1], On[:, :, -1]) and np.array_equal(Lc[:, :, -1], Ln[:, :, -1])
    # query 0 of 3 sits at position 9: it sees keys 0..9, i.e. not the last two
    O9, L9 = orc.attention_qk(q[:, :, :1], k[:, :, :10], v[:, :, :10], 0.4, False)
    assert np.abs(Oc[:, :, 0] - O9[:, :, 0]).max() < 1e-15


def pin_closed_form_first_causal_row(orc):
    """Causal row 0 sees key 0 only: O_0 = V_0 and LSE_0 = s_00."""
    q, k, v = inputs.attn_inputs(2, 3, 9, 8, seed=6)
    O, L = orc.attention(q, k, v, 0.25, True)
    qf, kf, vf = _bf16_float(q), _bf16_float(k), _bf16_float(v)
    assert np.array_equal(O[:, :, 0], vf[:, :, 0])
    s00 = 0.25 * np.einsum("bhk,bhk->bh", qf[:, :, 0], kf[:, :, 0])
    assert np.abs(L[:, :, 0] - s00).max() < 1e-13


def pin_closed_form_two_keys(orc):
    """Two keys: weight of key 0 is the logistic 1 / (1 + exp(s1 - s0))."""
    q, k, v = inputs.attn_inputs(1, 1, 2, 6, seed=8, qk_std=2.0)
    O, L = orc.attention(q, k, v, 0.7, False)
    qf, kf, vf = _bf16_float(q)[0, 0], _bf16_float(k)[0, 0], _bf16_float(v)[0, 0]
    for i in range(2):
        s0 = 0.7 * float(qf[i] @ kf[0])
        s1 = 0.7 * float(qf[i] @ kf[1])
        w0 = 1.0 / (1.0 + math.exp(s1 - s0))
        assert np.abs(O[0, 0, i] - (w0 * vf[0] + (1 - w0) * vf[1])).max() < 1e-14
        hi = max(s0, s1)
        assert abs(L[0, 0, i] - (hi + math.log1p(math.exp(-abs(s1 - s0))))) < 1e-13


def pin_closed_form_constant_values_and_zero_scale(orc):
    q, k, _ = inputs.attn_inputs(1, 2, 13, 4, seed=9, qk_std=3.0)
    v = torch.full((1, 2, 13, 4), 0.75).to(torch.bfloat16)
    O, _ = orc.attention(q, k, v, 0.5, True)
    assert np.abs(O - 0.75).max() < 1e-14
    q, k, v = inputs.attn_inputs(1, 1, 10, 4, seed=10)
    O, L = orc.attention(q, k, v, 0.0, False)
    assert np.abs(O[0, 0] - _bf16_float(v)[0, 0].mean(axis=0)).max() < 1e-14
    assert np.abs(L - math.log(10.0)).max() < 1e-14


# ----------------------------------------------------------------------------------------------
# invariants and laws
# ----------------------------------------------------------------------------------------------

def pin_shift_invariance(orc):
    """Adding one constant to every score of a row leaves O unchanged and moves LSE by it.
    Done by appending a feature: q' = [q, a], k'_j = [k_j, b] adds scale*a*b to every s_j."""
    q, k, v = inputs.attn_inputs(1, 2, 9, 3, seed=12)
    O, L = orc.attention(q, k, v, 0.5, False)
    a, b = 4.0, 8.0  # bf16-exact, shift = 0.5 * 32 = 16
    q4 = torch.cat([q, torch.full((1, 2, 9, 1), a).to(torch.bfloat16)], dim=-1)
    k4 = torch.cat([k, torch.full((1, 2, 9, 1), b).to(torch.bfloat16)], dim=-1)
    v4 = torch.cat([v, torch.zeros((1, 2, 9, 1)).to(torch.bfloat16)], dim=-1)
    O4, L4 = orc.attention(q4, k4, v4, 0.5, False)
    assert np.abs(O4[..., :3] - O).max() < 1e-14
    assert np.abs(L4 - (L + 16.0)).max() < 1e-12


def pin_key_permutation_invariance(orc):
    q, k, v = inputs.attn_inputs(1, 1, 12, 4, seed=13)
    perm = torch.randperm(12, generator=torch.Generator().manual_seed(3))
    O, L = orc.attention(q, k, v, 0.5, False)
    Op, Lp = orc.attention(q, k[:, :, perm], v[:, :, perm], 0.5, False)
    assert np.abs(O - Op).max() < 1e-14 and np.abs(L - Lp).max() < 1e-13
    Oq, _ = orc.attention(q[:, :, perm], k, v, 0.5, False)
    assert np.abs(Oq - O[:, :, perm.numpy()]).max() < 1e-14


def pin_block_size_independence(orc):
    """The streamed state at any block size gives the three-pass attention of that row."""
    N, d = 300, 16
    q, k, v = inputs.attn_inputs(1, 1, N, d, seed=14)
    O, L = orc.attention(q, k, v, 0.25, False, rows=np.array([0, 117, N - 1]))
    qf, kf, vf = _bf16_float(q)[0, 0], _bf16_float(k)[0, 0], _bf16_float(v)[0, 0]
    for r, i in enumerate([0, 117, N - 1]):
        s = 0.25 * (kf @ qf[i])
        for block in (1, 7, 64, 128, N):
            st = orc.online_state(s, vf, block=block)
            assert np.abs(st["acc"] / st["l"] - O[r]).max() < 1e-12, block
            assert abs(st["m"] + math.log(st["l"]) - L[r]) < 1e-12


def pin_merge_law(orc):
    """Two workers stream disjoint halves; merging their states equals one pass."""
    rng = np.random.default_rng(3)
    s, v = rng.normal(0, 3, size=100), rng.standard_normal((100, 8))
    whole = orc.online_state(s, v, block=10)
    left = orc.online_state(s[:37], v[:37], block=10)
    right = orc.online_state(s[37:], v[37:], block=10)
    for a, b in ((left, right), (right, left)):
        mg = orc.merge(a, b)
        assert abs(mg["m"] - whole["m"]) < 1e-15
        assert abs(mg["l"] - whole["l"]) < 1e-12 * whole["l"]
        assert np.abs(mg["acc"] - whole["acc"]).max() < 1e-12 * np.abs(whole["acc"]).max()
    empty = dict(m=-math.inf, l=0.0, acc=np.zeros(8))
    e = orc.merge(empty, left)
    assert e["l"] == left["l"] and np.array_equal(e["acc"], left["acc"])


def pin_softmax_rows_sum_to_one(orc):
    x = inputs.softmax_inputs(16, 1000, seed=15).numpy()
    y, lse = orc.softmax_rows(x)
    assert np.abs(y.sum(axis=1) - 1.0).max() < 1e-13
    assert np.all(y >= 0.0)
    # shift invariance of the softmax itself
    y2, lse2 = orc.softmax_rows(x + np.float32(3.0))
    assert np.abs(y2 - y).max() < 1e-6  # x + 3 is rounded to fp32 again
    assert np.abs(lse2 - lse - 3.0).max() < 1e-4


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]

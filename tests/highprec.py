"""Attention in 40-digit decimal arithmetic, by the textbook definition, for tiny inputs.

Pins the fp64 oracle to something other than itself: no max subtraction, no fp64 rounding,
softmax written as exp(s_j) / sum_k exp(s_k) exactly as the textbook formula of the
"FlashAttention Algorithm > Online Softmax Computation" page (mbrenndoerfer.com, the softmax
formula at the top) states it.  In decimal arithmetic the naive formula cannot overflow, so it
is exact to ~40 digits.  Pure-Python loops: keep the inputs tiny.
"""
from decimal import Decimal, getcontext

getcontext().prec = 40


def attention_decimal(q, K, V, scale, causal):
    """q, K, V: nested lists of Python floats (exact bf16 values), q [B][H][Nq][d] and
    K, V [B][H][Nk][d].  Causal: query i sees keys j <= i + Nk - Nq.

    Returns (O, LSE) as nested lists of floats.
    """
    sc = Decimal(scale)
    O, L = [], []
    for b in range(len(q)):
        Ob, Lb = [], []
        for h in range(len(q[b])):
            Qh, Kh, Vh = q[b][h], K[b][h], V[b][h]
            N = len(Qh)
            Nk = len(Kh)
            d = len(Qh[0])
            Oh, Lh = [], []
            for i in range(N):
                keys = range(min(Nk, i + Nk - N + 1)) if causal else range(Nk)
                e = []
                for j in keys:
                    s = sum(Decimal(Qh[i][k]) * Decimal(Kh[j][k]) for k in range(d)) * sc
                    e.append(s.exp())
                tot = sum(e)
                row = []
                for k in range(d):
                    num = sum(e[t] * Decimal(Vh[j][k]) for t, j in enumerate(keys))
                    row.append(float(num / tot))
                Oh.append(row)
                Lh.append(float(tot.ln()))
            Ob.append(Oh)
            Lb.append(Lh)
        O.append(Ob)
        L.append(Lb)
    return O, L


def attention_decimal_gqa(q, K, V, scale, causal, kv_lens=None, mask=None):
    """As attention_decimal, with K, V [B][H_kv][Nk][d] shared by the H query heads (query head
    h reads key/value head h // (H // H_kv)), optional key lengths per sequence (keys
    j >= kv_lens[b] take no part) and an optional mask[b][h][i][j] (false: key j takes no part
    for query i).  A row with no key left gets O = 0 and LSE = -inf.
    """
    sc = Decimal(scale)
    O, L = [], []
    for b in range(len(q)):
        H, H_kv = len(q[b]), len(K[b])
        Ob, Lb = [], []
        for h in range(H):
            Qh, Kh, Vh = q[b][h], K[b][h // (H // H_kv)], V[b][h // (H // H_kv)]
            N, Nk, d = len(Qh), len(Kh), len(Qh[0])
            Oh, Lh = [], []
            for i in range(N):
                keys = [j for j in range(Nk)
                        if (not causal or j <= i + Nk - N) and (kv_lens is None or j < kv_lens[b])
                        and (mask is None or mask[b][h][i][j])]
                if not keys:
                    Oh.append([0.0] * d)
                    Lh.append(float("-inf"))
                    continue
                e = [(sum(Decimal(Qh[i][k]) * Decimal(Kh[j][k]) for k in range(d)) * sc).exp()
                     for j in keys]
                tot = sum(e)
                Oh.append([float(sum(e[t] * Decimal(Vh[j][k]) for t, j in enumerate(keys)) / tot)
                           for k in range(d)])
                Lh.append(float(tot.ln()))
            Ob.append(Oh)
            Lb.append(Lh)
        O.append(Ob)
        L.append(Lb)
    return O, L

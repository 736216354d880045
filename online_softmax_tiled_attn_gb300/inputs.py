"""Seeded synthetic inputs shared by the CUDA path's tests, the bench and the oracle's tests.

This module holds none of the method's arithmetic: it only draws random numbers and names the
workloads.  Every tensor is drawn on the CPU from ``torch.Generator().manual_seed(seed)`` in
fp32 and rounded once, round-to-nearest-even, to bf16; the same bf16 tensor is given to both
the GPU library and the fp64 oracle.  Q, then K, then V are drawn from one generator.

Workloads (shapes are [B, H, N, d], row-major, d innermost):

====================  ==========================================================================
name                  recipe
====================  ==========================================================================
small_b1h1n256d64     B1 H1 N256 d64, Q/K/V iid N(0,1), non-causal
mha_b4h16n2048d64     B4 H16 N2048 d64, Q/K/V iid N(0,1), non-causal
causal_b2h32n8192     B2 H32 N8192 d128, Q/K/V iid N(0,1), causal
causal_b1h8n32768     B1 H8 N32768 d128, Q/K/V iid N(0,1), causal (checked on sampled rows)
ragged_b1h16n4000     B1 H16 N4000 d128, Q,K iid N(0, sd 3) (logit sd 9), V iid U(-1,1)
dense_b2h32n8192      B2 H32 N8192 d128, Q/K/V iid N(0,1), non-causal (the d=128 long-N case)
softmax_65536x4000    fp32 rows [65536, 4000], x = 9*N(0,1) and per row one entry +100 and one
                      entry -100 at seeded positions
decode_b8h32q1k32768  B8 H32, one query against 32768 cached keys, d128, N(0,1), non-causal
                      (the split-key path); seed 1007
softmax_topk_*        the softmax workload's rows with top-k selection: [65536, 4000] k = 8 (seed
                      1005, the same rows), vocabulary-sized [512, 131072] k = 32 (1011) and
                      k = 100 (1018)
gqa_*                 grouped key/value heads (H_kv < H) and per-sequence key lengths, N(0,1):
                      a causal prefill, a ragged-length batch and a grouped decode; seeds
                      1008-1010 (see GQA_WORKLOADS)
====================  ==========================================================================

Seeds: 1000 + the workload's index in the table above (1001 ... 1005 for the five attention
workloads in the order listed, 1006 for the non-causal d=128 case, 1005 again for the softmax
rows, which belong to the ragged/overflow stress workload).
"""
from __future__ import annotations

import functools
import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class AttnWorkload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    qk_std: float = 1.0
    v_dist: str = "normal"  # "normal" N(0,1) or "uniform" U(-1,1)
    sample_rows_per_head: int = 0  # >0: parity on this many seeded rows per head

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Algorithmic FLOP: 4*B*H*N^2*d (two N x N x d contractions), halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    @property
    def hbm_bytes(self) -> int:
        """Compulsory HBM traffic: read Q, K, V (bf16), write O (bf16) and LSE (fp32)."""
        n = self.B * self.H * self.N
        return 4 * n * self.d * 2 + n * 4


@dataclass(frozen=True)
class SoftmaxWorkload:
    name: str
    rows: int
    cols: int
    seed: int
    std: float = 9.0
    spike: float = 100.0

    @property
    def hbm_bytes(self) -> int:
        """Compulsory HBM traffic: read x once, write y once (fp32), write lse (fp32)."""
        return self.rows * self.cols * 8 + self.rows * 4


ATTN_WORKLOADS = {
    w.name: w
    for w in [
        AttnWorkload("small_b1h1n256d64", 1, 1, 256, 64, False, 1001),
        AttnWorkload("mha_b4h16n2048d64", 4, 16, 2048, 64, False, 1002),
        AttnWorkload("causal_b2h32n8192", 2, 32, 8192, 128, True, 1003),
        AttnWorkload("causal_b1h8n32768", 1, 8, 32768, 128, True, 1004, sample_rows_per_head=512),
        AttnWorkload("ragged_b1h16n4000", 1, 16, 4000, 128, False, 1005, qk_std=3.0,
                     v_dist="uniform"),
        AttnWorkload("dense_b2h32n8192", 2, 32, 8192, 128, False, 1006),
    ]
}

@dataclass(frozen=True)
class DecodeWorkload:
    """Nq queries against a cache of Nk keys (the split-key / Flash-Decoding case)."""

    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        return 4.0 * self.B * self.H * self.Nq * self.Nk * self.d

    @property
    def hbm_bytes(self) -> int:
        """Compulsory HBM traffic: read Q, K, V (bf16), write O (bf16) and LSE (fp32)."""
        bh = self.B * self.H
        return bh * (2 * self.Nq * self.d * 2 + 2 * self.Nk * self.d * 2 + self.Nq * 4)


DECODE_WORKLOADS = {
    w.name: w
    for w in [DecodeWorkload("decode_b8h32q1k32768d128", 8, 32, 1, 32768, 128, False, 1007)]
}


@dataclass(frozen=True)
class GqaWorkload:
    """Q [B, H, Nq, d] against K, V [B, H_kv, Nk, d], optional key lengths per sequence."""

    name: str
    B: int
    H: int
    H_kv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int
    kv_lens: tuple = None  # valid keys per sequence, or None (all Nk)
    n_splits: int = 1      # 0: the library chooses a key split

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def lens(self):
        return list(self.kv_lens) if self.kv_lens is not None else [self.Nk] * self.B

    def allowed_pairs(self) -> int:
        """Allowed (query, key) pairs of one head summed over the sequences: query i of
        sequence b sees min(kv_len_b, i + 1 + Nk - Nq) keys when causal, kv_len_b otherwise."""
        tot = 0
        for L in self.lens():
            if not self.causal:
                tot += self.Nq * L
                continue
            off = self.Nk - self.Nq
            for i in range(self.Nq):
                tot += max(0, min(L, i + 1 + off))
        return tot

    @property
    def flops(self) -> float:
        """Algorithmic FLOP: 4*d per allowed (query, key) pair, for every query head."""
        return 4.0 * self.d * self.H * self.allowed_pairs()

    @property
    def hbm_bytes(self) -> int:
        """Compulsory HBM traffic: Q and O (bf16), LSE (fp32), and the valid keys' K and V."""
        q = self.B * self.H * self.Nq
        kv = self.H_kv * sum(self.lens())
        return q * self.d * 2 * 2 + q * 4 + kv * self.d * 2 * 2


GQA_WORKLOADS = {
    w.name: w
    for w in [
        GqaWorkload("gqa_causal_b2h32kv8n8192d128", 2, 32, 8, 8192, 8192, 128, True, 1008),
        GqaWorkload("gqa_ragged_b4h32kv8n4096d128", 4, 32, 8, 4096, 4096, 128, False, 1009,
                    kv_lens=(4096, 3000, 1500, 577)),
        GqaWorkload("gqa_decode_b8h32kv8q1k32768d128", 8, 32, 8, 1, 32768, 128, False, 1010,
                    n_splits=0),
    ]
}


def gqa_inputs(w: GqaWorkload):
    """Q [B,H,Nq,d], K and V [B,H_kv,Nk,d], bf16 N(0,1), drawn in that order from one seeded
    generator."""
    g = torch.Generator().manual_seed(int(w.seed))
    q = torch.randn((w.B, w.H, w.Nq, w.d), generator=g).to(torch.bfloat16)
    k = torch.randn((w.B, w.H_kv, w.Nk, w.d), generator=g).to(torch.bfloat16)
    v = torch.randn((w.B, w.H_kv, w.Nk, w.d), generator=g).to(torch.bfloat16)
    return q, k, v


def decode_inputs(w: DecodeWorkload):
    """Q [B,H,Nq,d] and K, V [B,H,Nk,d], bf16 N(0,1), from one seeded generator."""
    g = torch.Generator().manual_seed(int(w.seed))
    q = torch.randn((w.B, w.H, w.Nq, w.d), generator=g).to(torch.bfloat16)
    k = torch.randn((w.B, w.H, w.Nk, w.d), generator=g).to(torch.bfloat16)
    v = torch.randn((w.B, w.H, w.Nk, w.d), generator=g).to(torch.bfloat16)
    return q, k, v


SOFTMAX_WORKLOADS = {
    w.name: w for w in [SoftmaxWorkload("softmax_65536x4000", 65536, 4000, 1005)]
}


@dataclass(frozen=True)
class BwdWorkload:
    """Gradients of attention over Q, K, V, dO [B, H, N, d] (O and LSE from the forward)."""

    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Algorithmic FLOP: 10*B*H*N^2*d (five N x N x d contractions: S, dP, dV, dK, dQ),
        halved when causal."""
        f = 10.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    @property
    def hbm_bytes(self) -> int:
        """Compulsory HBM traffic: read Q, K, V, O, dO (bf16) and LSE (fp32), write dQ, dK, dV
        (bf16)."""
        n = self.B * self.H * self.N
        return 8 * n * self.d * 2 + n * 4


BWD_WORKLOADS = {
    w.name: w
    for w in [
        BwdWorkload("bwd_b4h16n2048d64", 4, 16, 2048, 64, False, 1012),
        BwdWorkload("bwd_b2h16n8192d128", 2, 16, 8192, 128, False, 1013),
        BwdWorkload("bwd_causal_b2h16n8192d128", 2, 16, 8192, 128, True, 1014),
    ]
}


def bwd_inputs(B, H, N, d, seed):
    """Q, K, V, dO as CPU bf16 tensors [B, H, N, d], N(0,1), drawn in that order from one seeded
    generator."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (B, H, N, d)
    return tuple(torch.randn(shape, generator=g).to(torch.bfloat16) for _ in range(4))


def random_mask(B, H, Nq, Nk, density, seed, full_rows=0, full_keys=0):
    """A seeded attention mask, uint8 [B, H, Nq, Nk] (1 = allowed), each entry allowed with
    probability `density`; then `full_rows` seeded query rows of every (b, h) are masked
    entirely and `full_keys` seeded keys are masked for every query."""
    g = torch.Generator().manual_seed(int(seed))
    m = (torch.rand((B, H, Nq, Nk), generator=g) < density).to(torch.uint8)
    for _ in range(full_rows):
        m[:, :, int(torch.randint(Nq, (1,), generator=g)), :] = 0
    for _ in range(full_keys):
        m[:, :, :, int(torch.randint(Nk, (1,), generator=g))] = 0
    return m.numpy()


def window_mask(Nq, Nk, window, doc_len):
    """uint8 [1, 1, Nq, Nk]: query i sees key j when they lie in the same document of `doc_len`
    positions and j <= i < j + window (a sliding window inside documents)."""
    i = np.arange(Nq)[:, None]
    j = np.arange(Nk)[None, :]
    m = (j <= i) & (i < j + window) & (i // doc_len == j // doc_len)
    return m.astype(np.uint8)[None, None]


def pack_mask(mask):
    """The bit layout fa_fwd_mask reads: uint32 [Bm, Hm, Nq, W] with W = 4 * ceil(Nk / 128);
    bit j % 32 of word j // 32 of a row is entry j (1 = allowed); bits past Nk are 0."""
    m = np.asarray(mask) != 0
    Bm, Hm, Nq, Nk = m.shape
    W = 4 * ((Nk + 127) // 128)
    padded = np.zeros((Bm, Hm, Nq, W * 32), dtype=bool)
    padded[..., :Nk] = m
    bits = np.packbits(padded.reshape(Bm, Hm, Nq, W, 32), axis=-1, bitorder="little")
    return np.ascontiguousarray(bits.view(np.uint32).reshape(Bm, Hm, Nq, W))


@dataclass(frozen=True)
class MaskWorkload:
    """Attention over Q, K, V [B, H, N, d] (N(0,1), from attn_inputs with this seed) with an
    explicit mask: "prefix_lm" (keys before `prefix` seen by every query, the rest causally;
    one [1, 1, N, N] mask for all heads), "window" (query i sees keys i - window + 1 .. i; one
    mask for all heads) or "random" (each entry allowed with probability `density`, one mask
    per head, [1, H, N, N]).  tile_map: whether the call passes fa_fwd_mask a tile map (worth
    it where whole 128 x 128 tiles are masked)."""

    name: str
    B: int
    H: int
    N: int
    d: int
    seed: int
    kind: str
    prefix: int = 0
    density: float = 1.0
    window: int = 0
    tile_map: bool = True

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def mask(self):
        """uint8 [1, 1 or H, N, N], 1 = allowed (made once per workload and kept: read only)."""
        return _workload_mask(self)

    def _make_mask(self):
        if self.kind == "prefix_lm":
            i = np.arange(self.N)[:, None]
            j = np.arange(self.N)[None, :]
            return ((j < self.prefix) | (j <= i)).astype(np.uint8)[None, None]
        if self.kind == "window":
            i = np.arange(self.N)[:, None]
            j = np.arange(self.N)[None, :]
            return ((j <= i) & (j > i - self.window)).astype(np.uint8)[None, None]
        return random_mask(1, self.H, self.N, self.N, self.density, self.seed + 1)

    @property
    def flops(self) -> float:
        """Algorithmic FLOP: 4*d per allowed (query, key) pair, summed over every head."""
        m = self.mask()
        per_mask = float(np.count_nonzero(m))
        heads_per_mask = self.B * self.H / m.shape[1]
        return 4.0 * self.d * per_mask * heads_per_mask

    @property
    def hbm_bytes(self) -> int:
        """Compulsory HBM traffic: Q, K, V read and O written (bf16), LSE (fp32), the mask bits."""
        n = self.B * self.H * self.N
        m = self.mask()
        return 4 * n * self.d * 2 + n * 4 + m.shape[1] * self.N * (4 * ((self.N + 127) // 128)) * 4


@functools.lru_cache(maxsize=4)
def _workload_mask(w):
    m = w._make_mask()
    m.setflags(write=False)
    return m


MASK_WORKLOADS = {
    w.name: w
    for w in [
        MaskWorkload("mask_prefixlm_b2h16n4096d128", 2, 16, 4096, 128, 1015, "prefix_lm",
                     prefix=1024),
        MaskWorkload("mask_random_b2h16n4096d128", 2, 16, 4096, 128, 1016, "random",
                     density=0.9, tile_map=False),
        MaskWorkload("mask_window_b2h16n8192d128", 2, 16, 8192, 128, 1017, "window",
                     window=1024),
    ]
}


def attn_inputs(B, H, N, d, seed, qk_std=1.0, v_dist="normal"):
    """Q, K, V as CPU bf16 tensors [B, H, N, d] drawn from one seeded generator."""
    g = torch.Generator().manual_seed(int(seed))
    shape = (B, H, N, d)
    q = (torch.randn(shape, generator=g, dtype=torch.float32) * qk_std).to(torch.bfloat16)
    k = (torch.randn(shape, generator=g, dtype=torch.float32) * qk_std).to(torch.bfloat16)
    if v_dist == "normal":
        v = torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)
    elif v_dist == "uniform":
        v = (torch.rand(shape, generator=g, dtype=torch.float32) * 2.0 - 1.0).to(torch.bfloat16)
    else:
        raise ValueError(v_dist)
    return q, k, v


def workload_inputs(w: AttnWorkload):
    return attn_inputs(w.B, w.H, w.N, w.d, w.seed, w.qk_std, w.v_dist)


def sample_rows(w: AttnWorkload, per_head: int, seed_offset: int = 0):
    """Seeded flat row indices (b*H + h)*N + i, `per_head` distinct rows in every head.

    Row 0 and row N-1 of every head are always included (the causal first row and the ragged
    last row are the rows most likely to go wrong).
    """
    g = torch.Generator().manual_seed(int(w.seed) * 7919 + 17 + seed_offset)
    out = []
    k = min(per_head, w.N)
    for bh in range(w.B * w.H):
        idx = torch.randperm(w.N, generator=g)[:k]
        idx[0] = 0
        if k > 1:
            idx[1] = w.N - 1
        idx = torch.unique(idx)
        out.append(idx.to(torch.int64) + bh * w.N)
    return torch.cat(out).numpy()


@dataclass(frozen=True)
class TopkWorkload:
    """Softmax with top-k selection over fp32 rows drawn as the softmax workload's."""

    name: str
    rows: int
    cols: int
    k: int
    seed: int
    std: float = 9.0
    spike: float = 100.0

    @property
    def hbm_bytes(self) -> int:
        """Compulsory HBM traffic: read x once; write k shares (fp32) and columns (int32) and
        the lse (fp32) of every row."""
        return self.rows * self.cols * 4 + self.rows * (self.k * 8 + 4)


TOPK_WORKLOADS = {
    w.name: w
    for w in [
        TopkWorkload("softmax_topk_65536x4000_k8", 65536, 4000, 8, 1005),
        TopkWorkload("softmax_topk_512x131072_k32", 512, 131072, 32, 1011),
        # vocabulary-scale sampling with a wider candidate set (radix selection, k > 32)
        TopkWorkload("softmax_topk_512x131072_k100", 512, 131072, 100, 1018),
    ]
}


def softmax_inputs(rows, cols, seed, std=9.0, spike=100.0):
    """fp32 [rows, cols]: std * N(0,1), and per row one +spike and one -spike entry."""
    g = torch.Generator().manual_seed(int(seed))
    x = torch.randn((rows, cols), generator=g, dtype=torch.float32) * std
    if cols >= 2 and spike:
        pos = torch.randint(0, cols, (rows, 2), generator=g)
        pos[:, 1] = (pos[:, 0] + 1 + torch.randint(0, cols - 1, (rows,), generator=g)) % cols
        r = torch.arange(rows)
        x[r, pos[:, 0]] = spike
        x[r, pos[:, 1]] = -spike
    return x


def softmax_workload_inputs(w: SoftmaxWorkload):
    return softmax_inputs(w.rows, w.cols, w.seed, w.std, w.spike)


def bf16_bits(t: torch.Tensor):
    """uint16 numpy view of a CPU bf16 tensor (what the oracle reads)."""
    import numpy as np

    return t.contiguous().view(torch.int16).numpy().view(np.uint16)

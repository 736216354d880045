"""The C-ABI library builds, loads on a machine without a GPU, exports every function that
include/osm_attn.h declares, and rejects bad arguments on the host before any CUDA call."""
import ctypes
import os
import re

import pytest

from online_softmax_tiled_attn_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    names = []
    for f in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if f.endswith(".h"):
            text = open(os.path.join(ROOT, "include", f)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^\s*(?:OSM_ATTN_API\s+)?(?:const\s+)?\w+\s*\**\s*(\w+)\s*\(",
                                text, flags=re.M)
    return names


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_fwd", "fa_fwd_splitkv", "fa_fwd_splitkv_plan", "fa_fwd_gqa", "fa_fwd_gqa_plan",
              "osm_softmax", "osm_softmax_topk", "fa_bwd", "fa_fwd_mask", "fa_fwd_mask_plan",
              "fa_fwd_gqa_mask", "fa_fwd_gqa_mask_plan", "fa_bwd_gqa", "fa_fwd_host",
              "fa_status_string", "osm_attn_device_status", "osm_attn_selftest_wait",
              "osm_attn_abi_version"):
        assert n in names


def test_library_exports_every_declared_symbol_and_nothing_else():
    import subprocess

    L = binding.lib()
    for n in declared_functions():
        assert hasattr(L, n), n
        assert isinstance(getattr(L, n), ctypes._CFuncPtr)
    out = subprocess.run(["nm", "-D", "--defined-only", binding.build_lib.LIB],
                         capture_output=True, text=True)
    if out.returncode == 0:
        exported = {ln.split()[-1] for ln in out.stdout.splitlines() if " T " in ln}
        assert exported == set(declared_functions()), exported ^ set(declared_functions())


def test_status_strings_and_version():
    assert binding.status_string(0) == "FA_OK"
    for s in range(1, 5):
        assert binding.status_string(s).startswith("FA_ERR_")
    assert binding.status_string(99) == "unknown fa_status"
    assert binding.lib().osm_attn_abi_version() == 10


# A fake device address: every case below must be rejected on the host, before any launch,
# so it is never dereferenced.
P = 1 << 20


@pytest.mark.parametrize(
    "args, want",
    [
        ((P, P + 4096, P + 8192, P + 12288, 0, -1, 1, 128, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),
        ((P, P + 4096, P + 8192, P + 12288, 0, 1, 1, -5, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),
        ((0, 0, 0, 0, 0, 1, 1, 0, 64, 0.125, 0), binding.FA_OK),  # empty: no-op
        ((0, 0, 0, 0, 0, 0, 8, 128, 64, 0.125, 1), binding.FA_OK),  # B = 0: no-op
        ((P, P + 4096, P + 8192, P + 12288, 0, 1, 1, 128, 96, 0.125, 0), binding.FA_ERR_UNSUPPORTED),
        ((P, P + 4096, P + 8192, P + 12288, 0, 1, 1, 128, 32, 0.125, 0), binding.FA_ERR_UNSUPPORTED),
        ((0, P + 4096, P + 8192, P + 12288, 0, 1, 1, 128, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),
        ((P + 2, P + 65536, P + 131072, P + 196608, 0, 1, 1, 128, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),
        ((P, P + 65536, P + 131072, P + 196608, 0, 1, 1, 128, 64, float("nan"), 0), binding.FA_ERR_INVALID_ARG),
        ((P, P + 65536, P + 131072, P + 196608, 0, 1, 1, 128, 64, float("inf"), 0), binding.FA_ERR_INVALID_ARG),
        ((P, P + 65536, P + 131072, P + 196608, 0, 1, 1, 128, 64, 0.0, 0), binding.FA_ERR_INVALID_ARG),
        ((P, P + 65536, P + 131072, P + 196608, 0, 1, 1, 128, 64, -0.125, 0), binding.FA_ERR_INVALID_ARG),
        ((P, P + 65536, P + 131072, P, 0, 1, 1, 128, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),  # O == Q
        ((P, P + 65536, P + 131072, P + 131072 + 64, 0, 1, 1, 128, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),  # O overlaps V
        ((P, P + 65536, P + 131072, P + 196608, P + 196608 + 2, 1, 1, 128, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),  # LSE misaligned
        ((P, P + 65536, P + 131072, P + 196608, 0, 1 << 40, 1 << 40, 128, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),  # overflow
        ((P, P + 65536, P + 131072, P + 196608, P + 196608 + 4096, 1, 1, 128, 64, 0.125, 0), binding.FA_ERR_INVALID_ARG),  # LSE inside O
    ],
)
def test_fa_fwd_rejects_on_host(args, want):
    assert binding.fa_fwd_raw(*args, None) == want


@pytest.mark.parametrize(
    "args, want",
    [
        ((P, P, -1, 10, 0), binding.FA_ERR_INVALID_ARG),
        ((P, P, 10, -1, 0), binding.FA_ERR_INVALID_ARG),
        ((0, 0, 0, 10, 0), binding.FA_OK),
        ((0, 0, 10, 0, P), binding.FA_OK),
        ((0, P, 10, 10, 0), binding.FA_ERR_INVALID_ARG),
        ((P + 1, P + 8192, 10, 10, 0), binding.FA_ERR_INVALID_ARG),
        ((P, P + 8, 10, 10, 0), binding.FA_ERR_INVALID_ARG),  # partial overlap
        ((P, P + 8192, 1 << 40, 1 << 40, 0), binding.FA_ERR_INVALID_ARG),
    ],
)
def test_osm_softmax_rejects_on_host(args, want):
    assert binding.osm_softmax_raw(*args, None) == want


def test_fa_fwd_accepts_lse_just_below_an_input():
    """A small LSE buffer that ends right where Q starts does not overlap it.  The call passes
    validation and reaches the CUDA launch, which fails without a GPU (FA_ERR_CUDA), or
    succeeds with one; it is never FA_ERR_INVALID_ARG."""
    import torch

    if torch.cuda.is_available():
        pytest.skip("covered by the GPU tests on a machine with a GPU")
    B, H, N, d = 1, 1, 128, 64
    lse = P
    q = P + B * H * N * 4  # LSE [P, P + 512) ends where Q starts
    n = B * H * N * d * 2
    rc = binding.fa_fwd_raw(q, q + n, q + 2 * n, q + 3 * n, lse, B, H, N, d, 0.125, 0, None)
    assert rc == binding.FA_ERR_CUDA


# fa_fwd_gqa(Q, K, V, O, LSE, B, H, H_kv, Nq, Nk, d, scale, causal, kv_lens, n_splits, ...):
# B1 H4 Nq=Nk=128 d64; Q/O 64 KiB each, K/V sized by H_kv.
Q4 = 4 * 128 * 64 * 2


@pytest.mark.parametrize(
    "args, want",
    [
        ((P, P + Q4, P + 2 * Q4, P + 3 * Q4, 0, 1, 4, 3, 128, 128, 64, 0.125, 0, 0, 1),
         binding.FA_ERR_INVALID_ARG),  # H_kv does not divide H
        ((P, P + Q4, P + 2 * Q4, P + 3 * Q4, 0, 1, 4, 0, 128, 128, 64, 0.125, 0, 0, 1),
         binding.FA_ERR_INVALID_ARG),  # H_kv = 0
        ((P, P + Q4, P + 2 * Q4, P + 3 * Q4, 0, 1, 4, 2, 128, 128, 64, 0.125, 0, 0, 1),
         binding.FA_ERR_CUDA),  # valid: reaches the launch, which fails without a GPU
        ((P, P + Q4, P + 2 * Q4, P + 3 * Q4, 0, 1, 4, 2, 128, 128, 64, 0.125, 0, P + 5 * Q4 + 2,
          1), binding.FA_ERR_INVALID_ARG),  # kv_lens misaligned
        ((P, P + Q4, P + 2 * Q4, P + 3 * Q4, 0, 1, 4, 2, 128, 128, 64, 0.125, 0, P + 3 * Q4 + 64,
          1), binding.FA_ERR_INVALID_ARG),  # kv_lens inside O
        ((P, P + Q4, P + 2 * Q4, P + 3 * Q4, 0, 1, 4, 2, 128, 128, 64, 0.125, 0, 0, 0),
         binding.FA_ERR_INVALID_ARG),  # n_splits 0 is for the plan call, not this one
        ((P, P + Q4, P + 2 * Q4, P + 3 * Q4, 0, 1, 4, 2, 128, 128, 64, 0.125, 0, 0, 2),
         binding.FA_ERR_INVALID_ARG),  # two ranges without a workspace
        ((0, 0, 0, P, 0, 1, 4, 2, 128, 0, 64, 0.125, 0, 0, 1),
         binding.FA_ERR_CUDA),  # no key: the empty-row path, launched (fails without a GPU)
    ],
)
def test_fa_fwd_gqa_rejects_on_host(args, want):
    import torch

    if want == binding.FA_ERR_CUDA and torch.cuda.is_available():
        pytest.skip("reaches a launch; covered by the GPU tests on a machine with a GPU")
    assert binding.fa_fwd_gqa_raw(*args, None, None, None) == want


@pytest.mark.parametrize(
    "args, want",
    [
        ((P, -1, 10, 1, P + 4096, P + 8192, 0), binding.FA_ERR_INVALID_ARG),
        ((P, 10, 10, 0, P + 4096, P + 8192, 0), binding.FA_ERR_INVALID_ARG),   # k = 0
        ((P, 10, 10, 11, P + 4096, P + 8192, 0), binding.FA_ERR_INVALID_ARG),  # k > cols
        ((P, 10, 2000, 1025, P + 81920, P + 81920 + 65536, 0), binding.FA_ERR_UNSUPPORTED),  # k > 1024
        ((0, 0, 10, 4, 0, 0, 0), binding.FA_OK),                               # no rows
        ((0, 10, 10, 4, P + 4096, P + 8192, 0), binding.FA_ERR_INVALID_ARG),   # x null
        ((P + 2, 10, 10, 4, P + 4096, P + 8192, 0), binding.FA_ERR_INVALID_ARG),  # misaligned
        ((P, 10, 10, 4, P + 200, P + 8192, 0), binding.FA_ERR_INVALID_ARG),    # values in x
        ((P, 10, 10, 4, P + 4096, P + 4096 + 80, 0), binding.FA_ERR_INVALID_ARG),  # overlap
        ((P, 10, 10, 4, P + 4096, P + 8192, P + 8192 + 8), binding.FA_ERR_INVALID_ARG),
    ],
)
def test_osm_softmax_topk_rejects_on_host(args, want):
    assert binding.osm_softmax_topk_raw(*args, None) == want


def _bwd_args(**over):
    """fa_bwd arguments for B1 H1 N128 d64 at distinct fake addresses (16 KiB per tensor)."""
    T = 128 * 64 * 2
    a = dict(q=P, k=P + T, v=P + 2 * T, o=P + 3 * T, do=P + 4 * T, lse=P + 5 * T,
             dq=P + 6 * T, dk=P + 7 * T, dv=P + 8 * T, ws_d=P + 9 * T,
             B=1, H=1, N=128, d=64, scale=0.125, causal=0)
    a.update(over)
    return a


@pytest.mark.parametrize(
    "over, want",
    [
        (dict(N=-1), binding.FA_ERR_INVALID_ARG),
        (dict(N=0), binding.FA_OK),
        (dict(d=96), binding.FA_ERR_UNSUPPORTED),
        (dict(scale=0.0), binding.FA_ERR_INVALID_ARG),
        (dict(dq=0), binding.FA_ERR_INVALID_ARG),
        (dict(dk=P + 2), binding.FA_ERR_INVALID_ARG),          # misaligned
        (dict(dv=P + 64), binding.FA_ERR_INVALID_ARG),         # dV inside Q
        (dict(ws_d=P + 6 * 16384), binding.FA_ERR_INVALID_ARG),   # workspace on dQ
        (dict(ws_d=P + 5 * 16384), binding.FA_ERR_INVALID_ARG),   # workspace on LSE
        (dict(ws_d=P + 9 * 16384 + 2), binding.FA_ERR_INVALID_ARG),  # misaligned workspace
    ],
)
def test_fa_bwd_rejects_on_host(over, want):
    a = _bwd_args(**over)
    rc = binding.fa_bwd_raw(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"], a["dk"],
                            a["dv"], a["ws_d"], a["B"], a["H"], a["N"], a["d"], a["scale"],
                            a["causal"], None)
    assert rc == want


@pytest.mark.parametrize(
    "over, want",
    [
        (dict(mask=0), binding.FA_ERR_INVALID_ARG),               # no mask
        (dict(mask=P + 9 * 16384 + 4), binding.FA_ERR_INVALID_ARG),  # misaligned
        (dict(mbs=-4), binding.FA_ERR_INVALID_ARG),
        (dict(mhs=6), binding.FA_ERR_INVALID_ARG),                 # not whole 16-byte groups
        (dict(mask=P + 3 * 16384), binding.FA_ERR_INVALID_ARG),    # mask on O
        (dict(d=96), binding.FA_ERR_UNSUPPORTED),
        (dict(Nq=0), binding.FA_OK),
        (dict(tm=P + 11 * 16384 + 2, tmw=1), binding.FA_ERR_INVALID_ARG),  # tile map misaligned
        (dict(tm=P + 11 * 16384, tmw=0), binding.FA_ERR_INVALID_ARG),      # tile map too small
        (dict(tm=P + 3 * 16384, tmw=1), binding.FA_ERR_INVALID_ARG),       # tile map on O
        (dict(tm=P + 9 * 16384 + 64, tmw=1), binding.FA_ERR_INVALID_ARG),  # tile map on the mask
        (dict(tm=P, tmw=1), binding.FA_ERR_INVALID_ARG),                   # tile map on Q
    ],
)
def test_fa_fwd_mask_rejects_on_host(over, want):
    """B1 H1 N128 d64 at distinct fake addresses (16 KiB per tensor), mask at the tenth."""
    T = 128 * 64 * 2
    a = dict(q=P, k=P + T, v=P + 2 * T, o=P + 3 * T, lse=P + 4 * T, B=1, H=1, Nq=128, Nk=128,
             d=64, scale=0.125, causal=0, mask=P + 9 * T, mbs=0, mhs=0, tm=0, tmw=0)
    a.update(over)
    rc = binding.fa_fwd_mask_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                 a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"], a["mask"],
                                 a["mbs"], a["mhs"], a["tm"], a["tmw"], None)
    assert rc == want


def test_fa_fwd_mask_plan_sizes():
    """One row of ceil(key tiles / 32) words per 128-row query tile and mask instance."""
    assert binding.mask_plan(1, 1, 128, 128, 0, 0) == 1
    assert binding.mask_plan(2, 16, 4096, 4096, 0, 0) == 32            # one shared mask
    assert binding.mask_plan(2, 16, 4096, 4096, 0, 4096 * 128) == 16 * 32   # per head
    assert binding.mask_plan(2, 16, 4096, 4096, 16 * 4096 * 128, 4096 * 128) == 2 * 16 * 32
    assert binding.mask_plan(2, 16, 4096, 4096, 16 * 4096 * 128, 0) == 2 * 32  # per sequence
    assert binding.mask_plan(1, 1, 300, 5000, 0, 0) == 3 * 2           # 40 key tiles: 2 words
    assert binding.mask_plan(1, 1, 0, 5000, 0, 0) == 0
    for bad in ((-1, 1, 128, 128, 0, 0), (1, 1, 128, 128, -4, 0), (1, 1, 1 << 31, 128, 0, 0)):
        with pytest.raises(binding.FaError):
            binding.mask_plan(*bad)


@pytest.mark.parametrize(
    "over, want",
    [
        (dict(mask=0), binding.FA_ERR_INVALID_ARG),                  # no mask
        (dict(Hkv=3), binding.FA_ERR_INVALID_ARG),                   # H_kv does not divide H
        (dict(mhs=6), binding.FA_ERR_INVALID_ARG),                   # not whole 16-byte groups
        (dict(lens=P + 3 * 65536 + 64), binding.FA_ERR_INVALID_ARG),  # key lengths inside O
        (dict(splits=2), binding.FA_ERR_INVALID_ARG),                # two ranges, no workspace
        (dict(splits=2, wso=P + 12 * 65536, wsl=P + 12 * 65536 + 8), binding.FA_ERR_INVALID_ARG),
        (dict(splits=0), binding.FA_ERR_INVALID_ARG),                # 0 is for the plan call
        (dict(tm=P + 3 * 65536, tmw=1), binding.FA_ERR_INVALID_ARG),  # tile map on O
        (dict(d=96), binding.FA_ERR_UNSUPPORTED),
        (dict(Nq=0), binding.FA_OK),
    ],
)
def test_fa_fwd_gqa_mask_rejects_on_host(over, want):
    """B1 H4 H_kv 2 Nq=Nk=128 d64 at distinct fake addresses (64 KiB slots), mask at the tenth."""
    T = 65536
    a = dict(q=P, k=P + T, v=P + 2 * T, o=P + 3 * T, lse=P + 4 * T, B=1, H=4, Hkv=2, Nq=128,
             Nk=128, d=64, scale=0.125, causal=0, lens=0, mask=P + 9 * T, mbs=0, mhs=0, tm=0,
             tmw=0, splits=1, wso=0, wsl=0)
    a.update(over)
    rc = binding.fa_fwd_gqa_mask_raw(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                                     a["Hkv"], a["Nq"], a["Nk"], a["d"], a["scale"], a["causal"],
                                     a["lens"], a["mask"], a["mbs"], a["mhs"], a["tm"], a["tmw"],
                                     a["splits"], a["wso"], a["wsl"], None)
    assert rc == want


def test_fa_fwd_gqa_mask_plan():
    """The tile map as fa_fwd_mask_plan; split counts over the unpacked query heads; the
    workspaces sized for the chosen count."""
    s, wo, wl, tm = binding.gqa_mask_plan(2, 16, 4, 4096, 4096, 128, 0, 4096 * 128, 3)
    assert s == 3 and wo == 3 * 2 * 16 * 4096 * 128 and wl == 3 * 2 * 16 * 4096
    assert tm == binding.mask_plan(2, 16, 4096, 4096, 0, 4096 * 128)
    s, wo, wl, tm = binding.gqa_mask_plan(1, 8, 8, 300, 5000, 64, 0, 0, 1)
    assert (s, wo, wl, tm) == (1, 0, 0, binding.mask_plan(1, 8, 300, 5000, 0, 0))
    s, _, _, _ = binding.gqa_mask_plan(1, 1, 1, 128, 300, 64, 0, 0, 64)
    assert s == 3  # capped at the key tiles
    for bad in ((1, 4, 3, 128, 128, 64, 0, 0, 0), (1, 4, 2, 128, 128, 64, -4, 0, 0),
                (1, 4, 2, 128, 128, 64, 0, 0, 300)):
        with pytest.raises(binding.FaError):
            binding.gqa_mask_plan(*bad)


@pytest.mark.parametrize(
    "over, want",
    [
        (dict(Hkv=3), binding.FA_ERR_INVALID_ARG),                  # H_kv does not divide H
        (dict(Hkv=0), binding.FA_ERR_INVALID_ARG),
        (dict(lens=P + 20 * 65536 + 2), binding.FA_ERR_INVALID_ARG),  # misaligned lengths
        (dict(dk=P + 20 * 65536 - 32), binding.FA_ERR_INVALID_ARG),  # dK reaches the lengths
        (dict(dv=P + 64), binding.FA_ERR_INVALID_ARG),               # dV inside Q
        (dict(N=0), binding.FA_OK),
        (dict(d=96), binding.FA_ERR_UNSUPPORTED),
    ],
)
def test_fa_bwd_gqa_rejects_on_host(over, want):
    """B1 H4 H_kv 2 N128 d64 at distinct fake addresses (64 KiB slots), lengths at the 21st."""
    T = 65536
    a = dict(q=P, k=P + T, v=P + 2 * T, o=P + 3 * T, do=P + 4 * T, lse=P + 5 * T, dq=P + 6 * T,
             dk=P + 7 * T, dv=P + 8 * T, ws=P + 9 * T, B=1, H=4, Hkv=2, N=128, d=64, scale=0.125,
             causal=0, lens=P + 20 * T)
    a.update(over)
    rc = binding.fa_bwd_gqa_raw(a["q"], a["k"], a["v"], a["o"], a["do"], a["lse"], a["dq"],
                                a["dk"], a["dv"], a["ws"], a["B"], a["H"], a["Hkv"], a["N"],
                                a["d"], a["scale"], a["causal"], a["lens"], None)
    assert rc == want


@pytest.mark.parametrize("over,want", [
    (dict(qh=0), binding.FA_ERR_INVALID_ARG),                  # NULL host input
    (dict(oh=0), binding.FA_ERR_INVALID_ARG),                  # NULL host output
    (dict(lh=0), binding.FA_ERR_INVALID_ARG),                  # LSE on the device only
    (dict(ld=0), binding.FA_ERR_INVALID_ARG),                  # LSE on the host only
    (dict(kd=P + 8 * 65536 + 32), binding.FA_ERR_INVALID_ARG),  # K staging overlaps O staging
    (dict(ld=P + 5 * 65536 + 64), binding.FA_ERR_INVALID_ARG),  # LSE staging inside V staging
    (dict(vd=P + 6 * 65536 + 8), binding.FA_ERR_INVALID_ARG),  # misaligned staging
    (dict(d=96), binding.FA_ERR_UNSUPPORTED),
    (dict(scale=0.0), binding.FA_ERR_INVALID_ARG),
    (dict(chunks=-1), binding.FA_ERR_INVALID_ARG),
    (dict(chunks=65), binding.FA_ERR_INVALID_ARG),
    (dict(N=0), binding.FA_OK),                                 # empty: nothing enqueued
])
def test_fa_fwd_host_rejects_on_host(over, want):
    """B1 H2 N128 d64 (32 KiB per tensor) at distinct fake addresses (64 KiB slots)."""
    T = 65536
    a = dict(qh=P, kh=P + T, vh=P + 2 * T, oh=P + 3 * T, lh=P + 4 * T, qd=P + 5 * T,
             kd=P + 6 * T, vd=P + 7 * T, od=P + 8 * T, ld=P + 9 * T, B=1, H=2, N=128, d=64,
             scale=0.125, chunks=0)
    a.update(over)
    # the LSE staging test above places LSE inside V's staging slot
    if over.get("ld") == P + 5 * T + 64:
        a["vd"] = P + 5 * T
        a["qd"] = P + 11 * T
    rc = binding.fa_fwd_host_raw(a["qh"] or None, a["kh"], a["vh"], a["oh"] or None,
                                 a["lh"] or None, a["qd"], a["kd"], a["vd"], a["od"],
                                 a["ld"] or None, a["B"], a["H"], a["N"], a["d"], a["scale"],
                                 0, a["chunks"], None)
    assert rc == want


def test_selftest_rejects_out_of_range_timeout_on_host():
    L = binding.lib()
    assert L.osm_attn_selftest_wait(0, None) == binding.FA_ERR_INVALID_ARG
    assert L.osm_attn_selftest_wait(10_000_001, None) == binding.FA_ERR_INVALID_ARG

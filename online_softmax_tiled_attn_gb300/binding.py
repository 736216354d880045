"""ctypes binding of libosmattn.so: the same entry points as include/osm_attn.h.

Argument marshalling only: every step of the computation runs in the CUDA library.  PyTorch is
used for device memory and streams.  There is no fallback: if the library cannot be built or
loaded, or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

from . import build_lib

FA_OK = 0
FA_ERR_INVALID_ARG = 1
FA_ERR_UNSUPPORTED = 2
FA_ERR_CUDA = 3
FA_ERR_TIMEOUT = 4
FA_ERR_SCRATCH_LIMIT = 5

_lock = threading.Lock()
_lib = None


class FaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """Load libosmattn.so (building it in-tree with nvcc first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = build_lib.LIB
            if not build_lib.up_to_date():
                path = build_lib.build()
            if not os.path.exists(path):
                raise RuntimeError(f"CUDA library {path} is missing")
            L = ctypes.CDLL(path)
            vp, i64 = ctypes.c_void_p, ctypes.c_int64
            L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, ctypes.c_float,
                                 ctypes.c_int, vp]
            L.fa_fwd.restype = ctypes.c_int
            L.fa_fwd_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64,
                                      i64, ctypes.c_float, ctypes.c_int, i64, vp]
            L.fa_fwd_host.restype = ctypes.c_int
            L.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                         ctypes.c_float, ctypes.c_int, i64, vp, vp, vp]
            L.fa_fwd_splitkv.restype = ctypes.c_int
            L.fa_fwd_splitkv_noalloc.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                                 ctypes.c_float, ctypes.c_int, i64, vp]
            L.fa_fwd_splitkv_noalloc.restype = ctypes.c_int
            L.fa_fwd_gqa.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                     ctypes.c_float, ctypes.c_int, vp, i64, vp, vp, vp]
            L.fa_fwd_gqa.restype = ctypes.c_int
            L.fa_fwd_gqa_plan.argtypes = [i64, i64, i64, i64, i64, i64, i64,
                                          ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_int64)]
            L.fa_fwd_gqa_plan.restype = ctypes.c_int
            i64p = ctypes.POINTER(ctypes.c_int64)
            L.fa_fwd_splitkv_plan.argtypes = [i64, i64, i64, i64, i64, i64, i64p, i64p, i64p]
            L.fa_fwd_splitkv_plan.restype = ctypes.c_int
            L.osm_softmax.argtypes = [vp, vp, i64, i64, vp, vp]
            L.osm_softmax.restype = ctypes.c_int
            L.fa_fwd_mask.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64,
                                      ctypes.c_float, ctypes.c_int, vp, i64, i64, vp, i64, vp]
            L.fa_fwd_mask.restype = ctypes.c_int
            L.fa_fwd_mask_plan.argtypes = [i64, i64, i64, i64, i64, i64, i64p]
            L.fa_fwd_mask_plan.restype = ctypes.c_int
            L.fa_fwd_gqa_mask.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, i64, i64,
                                          ctypes.c_float, ctypes.c_int, vp, vp, i64, i64, vp, i64,
                                          i64, vp, vp, vp]
            L.fa_fwd_gqa_mask.restype = ctypes.c_int
            L.fa_fwd_gqa_mask_plan.argtypes = [i64, i64, i64, i64, i64, i64, i64, i64, i64, i64p,
                                               i64p, i64p, i64p]
            L.fa_fwd_gqa_mask_plan.restype = ctypes.c_int
            L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                 ctypes.c_float, ctypes.c_int, vp]
            L.fa_bwd.restype = ctypes.c_int
            L.fa_bwd_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i64,
                                     i64, ctypes.c_float, ctypes.c_int, vp, vp]
            L.fa_bwd_gqa.restype = ctypes.c_int
            L.osm_softmax_topk.argtypes = [vp, i64, i64, i64, vp, vp, vp, vp]
            L.osm_softmax_topk.restype = ctypes.c_int
            L.fa_status_string.argtypes = [ctypes.c_int]
            L.fa_status_string.restype = ctypes.c_char_p
            L.osm_attn_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int)]
            L.osm_attn_device_status.restype = ctypes.c_int
            L.osm_attn_selftest_wait.argtypes = [i64, vp]
            L.osm_attn_selftest_wait.restype = ctypes.c_int
            L.osm_attn_abi_version.argtypes = []
            L.osm_attn_abi_version.restype = ctypes.c_int
            _lib = L
        return _lib


def status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(int(stream.cuda_stream))


# ------------------------------------------------------------------------------------------
# raw entry points (integers for pointers): the C ABI as is
# ------------------------------------------------------------------------------------------
def fa_fwd_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, N, d, scale, causal, stream_ptr):
    return lib().fa_fwd(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(N), int(d),
                        float(scale), int(bool(causal)), stream_ptr)


def fa_fwd_host_raw(qh, kh, vh, oh, lseh, qd, kd, vd, od, lsed, B, H, N, d, scale, causal,
                    n_chunks, stream_ptr):
    return lib().fa_fwd_host(qh, kh, vh, oh, lseh, qd, kd, vd, od, lsed, int(B), int(H),
                             int(N), int(d), float(scale), int(bool(causal)), int(n_chunks),
                             stream_ptr)


def fa_fwd_splitkv_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d, scale, causal,
                       n_splits, ws_o_ptr, ws_lse_ptr, stream_ptr):
    return lib().fa_fwd_splitkv(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(Nq),
                                int(Nk), int(d), float(scale), int(bool(causal)), int(n_splits),
                                ws_o_ptr, ws_lse_ptr, stream_ptr)


def fa_fwd_gqa_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, H_kv, Nq, Nk, d, scale, causal,
                   kv_lens_ptr, n_splits, ws_o_ptr, ws_lse_ptr, stream_ptr):
    return lib().fa_fwd_gqa(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(H_kv),
                            int(Nq), int(Nk), int(d), float(scale), int(bool(causal)),
                            kv_lens_ptr, int(n_splits), ws_o_ptr, ws_lse_ptr, stream_ptr)


def fa_fwd_splitkv_noalloc_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, Nq, Nk, d, scale,
                               causal, n_splits, stream_ptr):
    """The split-key attention with its partial states in the library's fixed scratch array
    (no workspace argument, no allocation)."""
    return lib().fa_fwd_splitkv_noalloc(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H),
                                        int(Nq), int(Nk), int(d), float(scale),
                                        int(bool(causal)), int(n_splits), stream_ptr)


def splitkv_plan(B, H, Nq, Nk, d, n_splits=0):
    """(splits, workspace O floats, workspace LSE floats) for fa_fwd_splitkv."""
    s, wo, wl = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    rc = lib().fa_fwd_splitkv_plan(int(B), int(H), int(Nq), int(Nk), int(d), int(n_splits),
                                   ctypes.byref(s), ctypes.byref(wo), ctypes.byref(wl))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv_plan")
    return s.value, wo.value, wl.value


def gqa_plan(B, H, H_kv, Nq, Nk, d, n_splits=0):
    """(splits, workspace O floats, workspace LSE floats) for fa_fwd_gqa."""
    s, wo, wl = ctypes.c_int64(0), ctypes.c_int64(0), ctypes.c_int64(0)
    rc = lib().fa_fwd_gqa_plan(int(B), int(H), int(H_kv), int(Nq), int(Nk), int(d),
                               int(n_splits), ctypes.byref(s), ctypes.byref(wo), ctypes.byref(wl))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_gqa_plan")
    return s.value, wo.value, wl.value


def osm_softmax_raw(x_ptr, y_ptr, rows, cols, lse_ptr, stream_ptr):
    return lib().osm_softmax(x_ptr, y_ptr, int(rows), int(cols), lse_ptr, stream_ptr)


def fa_fwd_mask_raw(q, k, v, o, lse, B, H, Nq, Nk, d, scale, causal, mask, mask_b_stride,
                    mask_h_stride, tile_map, tile_map_words, stream_ptr):
    return lib().fa_fwd_mask(q, k, v, o, lse, int(B), int(H), int(Nq), int(Nk), int(d),
                             float(scale), int(bool(causal)), mask, int(mask_b_stride),
                             int(mask_h_stride), tile_map, int(tile_map_words), stream_ptr)


def gqa_mask_plan(B, H, H_kv, Nq, Nk, d, mask_b_stride, mask_h_stride, n_splits=0):
    """(splits, workspace O floats, workspace LSE floats, tile map words) for fa_fwd_gqa_mask."""
    s, wo, wl, tm = (ctypes.c_int64(0) for _ in range(4))
    rc = lib().fa_fwd_gqa_mask_plan(int(B), int(H), int(H_kv), int(Nq), int(Nk), int(d),
                                    int(mask_b_stride), int(mask_h_stride), int(n_splits),
                                    ctypes.byref(s), ctypes.byref(wo), ctypes.byref(wl),
                                    ctypes.byref(tm))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_gqa_mask_plan")
    return s.value, wo.value, wl.value, tm.value


def fa_fwd_gqa_mask_raw(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, B, H, H_kv, Nq, Nk, d, scale,
                        causal, kv_lens_ptr, mask_ptr, mask_b_stride, mask_h_stride, tm_ptr,
                        tm_words, n_splits, ws_o_ptr, ws_lse_ptr, stream_ptr):
    return lib().fa_fwd_gqa_mask(q_ptr, k_ptr, v_ptr, o_ptr, lse_ptr, int(B), int(H), int(H_kv),
                                 int(Nq), int(Nk), int(d), float(scale), int(bool(causal)),
                                 kv_lens_ptr, mask_ptr, int(mask_b_stride), int(mask_h_stride),
                                 tm_ptr, int(tm_words), int(n_splits), ws_o_ptr, ws_lse_ptr,
                                 stream_ptr)


def mask_plan(B, H, Nq, Nk, mask_b_stride, mask_h_stride):
    """Words of fa_fwd_mask's tile map for this shape and these mask strides."""
    w = ctypes.c_int64(0)
    rc = lib().fa_fwd_mask_plan(int(B), int(H), int(Nq), int(Nk), int(mask_b_stride),
                                int(mask_h_stride), ctypes.byref(w))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_mask_plan")
    return w.value


def fa_bwd_raw(q, k, v, o, do, lse, dq, dk, dv, ws_d, B, H, N, d, scale, causal, stream_ptr):
    return lib().fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws_d, int(B), int(H), int(N), int(d),
                        float(scale), int(bool(causal)), stream_ptr)


def osm_softmax_topk_raw(x_ptr, rows, cols, k, values_ptr, indices_ptr, lse_ptr, stream_ptr):
    return lib().osm_softmax_topk(x_ptr, int(rows), int(cols), int(k), values_ptr, indices_ptr,
                                  lse_ptr, stream_ptr)


def selftest_wait(timeout_us: int, stream=None) -> None:
    """Launch the bounded-wait diagnostic (a wait that nothing completes gives up after
    timeout_us and records FA_ERR_TIMEOUT for device_status to report)."""
    rc = lib().osm_attn_selftest_wait(int(timeout_us), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "osm_attn_selftest_wait")


def device_status(stream=None) -> int:
    """Synchronise `stream` and read/clear the kernels' bounded-wait status word."""
    st = ctypes.c_int(0)
    rc = lib().osm_attn_device_status(_stream_handle(stream), ctypes.byref(st))
    if rc != FA_OK:
        raise FaError(rc, "osm_attn_device_status")
    return st.value


# ------------------------------------------------------------------------------------------
# torch-tensor wrappers
# ------------------------------------------------------------------------------------------
def fa_fwd(q, k, v, scale=None, causal=False, out=None, lse=None, return_lse=True,
           stream=None):
    """O, LSE = attention(q, k, v) for CUDA bf16 tensors [B, H, N, d] (d = 64 or 128).

    scale defaults to 1/sqrt(d).  `out` ([B,H,N,d] bf16) and `lse` ([B,H,N] fp32) may be
    given to write into; with return_lse=False and no `lse`, LSE is not computed.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 [B, H, N, d] tensor")
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    elif out.shape != q.shape or out.dtype != torch.bfloat16 or not out.is_contiguous():
        raise TypeError("out must be a contiguous bf16 tensor shaped like q")
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None and (lse.dtype != torch.float32 or lse.numel() != B * H * N
                            or not lse.is_contiguous()):
        raise TypeError("lse must be a contiguous fp32 tensor of B*H*N elements")
    rc = fa_fwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                    lse.data_ptr() if lse is not None else None, B, H, N, d, scale, causal,
                    _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return out, lse


def fa_fwd_host(q, k, v, scale=None, causal=False, out=None, lse=None, return_lse=True,
                staging=None, n_chunks=0, stream=None):
    """O, LSE = attention(q, k, v) for host (CPU) bf16 tensors [B, H, N, d]: the library copies
    groups of heads to the device, runs the attention and copies O and LSE back, the copies
    overlapped with the attention.  q, k, v and `out`/`lse` (host, made page-locked here when
    not given) should be page-locked for the overlap.  `staging` may be the device tensors
    (q_dev, k_dev, v_dev, o_dev, lse_dev or None); otherwise they are allocated here on the
    current CUDA device.  Enqueued on `stream` (the current stream by default); the results are
    ready once it is synchronised, which this function does before it returns."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.is_cuda:
            raise TypeError(f"{name} must be a host (CPU) tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 [B, H, N, d] tensor")
    if q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k and v must share one [B, H, N, d] shape")
    B, H, N, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    if lse is None and return_lse:
        lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    for name, t, dt, n in (("out", out, torch.bfloat16, q.numel()),
                           ("lse", lse, torch.float32, B * H * N)):
        if t is not None and (t.is_cuda or t.dtype != dt or t.numel() != n
                              or not t.is_contiguous()):
            raise TypeError(f"{name} must be a contiguous host tensor of {n} {dt} elements")
    if staging is None:
        dev = torch.device("cuda", torch.cuda.current_device())
        qd = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
        staging = (qd, torch.empty_like(qd), torch.empty_like(qd), torch.empty_like(qd),
                   torch.empty((B, H, N), dtype=torch.float32, device=dev)
                   if lse is not None else None)
    qd, kd, vd, od, ld = staging
    for t in (qd, kd, vd, od):
        if not t.is_cuda or t.dtype != torch.bfloat16 or t.numel() != q.numel():
            raise TypeError("staging must hold four CUDA bf16 tensors shaped like q")
    if (ld is None) != (lse is None):
        raise TypeError("staging's LSE tensor must be given exactly when lse is")
    s = _stream_handle(stream)
    rc = fa_fwd_host_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr() if lse is not None else None, qd.data_ptr(),
                         kd.data_ptr(), vd.data_ptr(), od.data_ptr(),
                         ld.data_ptr() if ld is not None else None, B, H, N, d, scale, causal,
                         n_chunks, s)
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_host")
    (stream if stream is not None else torch.cuda.current_stream()).synchronize()
    return out, lse


def fa_fwd_splitkv(q, k, v, n_splits=0, scale=None, causal=False, out=None, lse=None,
                   return_lse=True, workspace=None, stream=None):
    """Attention of q [B,H,Nq,d] against k, v [B,H,Nk,d] (CUDA bf16) with the keys split into
    key ranges computed in parallel and combined (Flash-Decoding).  n_splits = 0 lets the
    library choose.  `workspace` may be a (ws_O, ws_LSE) pair of fp32 CUDA tensors; otherwise
    it is allocated here (the library itself never allocates).  Returns (O, LSE)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 [B, H, N, d] tensor")
    if k.shape != v.shape or q.shape[:2] != k.shape[:2] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H,Nk,d] disagree")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    splits, wo, wl = splitkv_plan(B, H, Nq, Nk, d, n_splits)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws_o = ws_l = None
    if splits > 1:
        if workspace is None:
            ws_o = torch.empty(wo, dtype=torch.float32, device=q.device)
            ws_l = torch.empty(wl, dtype=torch.float32, device=q.device)
        else:
            ws_o, ws_l = workspace
            if ws_o.numel() < wo or ws_l.numel() < wl:
                raise ValueError("workspace too small for this split count")
    rc = fa_fwd_splitkv_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d, scale,
                            causal, max(splits, 1) if Nk > 0 else 0,
                            ws_o.data_ptr() if ws_o is not None else None,
                            ws_l.data_ptr() if ws_l is not None else None, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_splitkv")
    return out, lse


def fa_fwd_gqa(q, k, v, kv_lens=None, n_splits=1, scale=None, causal=False, out=None, lse=None,
               return_lse=True, workspace=None, stream=None):
    """Attention of q [B,H,Nq,d] against k, v [B,H_kv,Nk,d] (CUDA bf16; H_kv divides H, query
    head h reads key/value head h // (H // H_kv)), with optional per-sequence key lengths
    kv_lens (CUDA int32 [B]: keys at or past kv_lens[b] are masked).  n_splits = 1 runs one
    pass; 0 lets the library choose a key split (Flash-Decoding), with a workspace allocated
    here unless `workspace` = (ws_O, ws_LSE) is given.  Returns (O, LSE)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 [B, H, N, d] tensor")
    if k.shape != v.shape or q.shape[0] != k.shape[0] or q.shape[3] != k.shape[3]:
        raise ValueError("q [B,H,Nq,d] and k, v [B,H_kv,Nk,d] disagree")
    B, H, Nq, d = q.shape
    H_kv, Nk = k.shape[1], k.shape[2]
    if kv_lens is not None:
        if not isinstance(kv_lens, torch.Tensor) or not kv_lens.is_cuda or \
                kv_lens.dtype != torch.int32 or kv_lens.shape != (B,) or \
                not kv_lens.is_contiguous():
            raise TypeError("kv_lens must be a contiguous CUDA int32 tensor of shape [B]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    splits, wo, wl = gqa_plan(B, H, H_kv, Nq, Nk, d, n_splits)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    ws_o = ws_l = None
    if splits > 1:
        if workspace is None:
            ws_o = torch.empty(wo, dtype=torch.float32, device=q.device)
            ws_l = torch.empty(wl, dtype=torch.float32, device=q.device)
        else:
            ws_o, ws_l = workspace
            if ws_o.numel() < wo or ws_l.numel() < wl:
                raise ValueError("workspace too small for this split count")
    rc = fa_fwd_gqa_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                        lse.data_ptr() if lse is not None else None, B, H, H_kv, Nq, Nk, d, scale,
                        causal, kv_lens.data_ptr() if kv_lens is not None else None,
                        max(splits, 1) if Nk > 0 else 0,
                        ws_o.data_ptr() if ws_o is not None else None,
                        ws_l.data_ptr() if ws_l is not None else None, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_gqa")
    return out, lse


def osm_softmax(x, out=None, lse=None, return_lse=True, stream=None):
    """y, lse = softmax of every row of a CUDA fp32 tensor [rows, cols] (out may be x)."""
    import torch

    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32:
        raise TypeError("x must be a CUDA fp32 tensor")
    if x.dim() != 2 or not x.is_contiguous():
        raise TypeError("x must be a contiguous [rows, cols] tensor")
    rows, cols = x.shape
    if out is None:
        out = torch.empty_like(x)
    elif out.shape != x.shape or out.dtype != torch.float32 or not out.is_contiguous():
        raise TypeError("out must be a contiguous fp32 tensor shaped like x")
    if lse is None and return_lse:
        lse = torch.empty((rows,), dtype=torch.float32, device=x.device)
    rc = osm_softmax_raw(x.data_ptr(), out.data_ptr(), rows, cols,
                         lse.data_ptr() if lse is not None else None, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "osm_softmax")
    return out, lse


def osm_softmax_topk(x, k, values=None, indices=None, lse=None, return_lse=True, stream=None):
    """(values, indices, lse): the k largest entries of every row of a CUDA fp32 [rows, cols]
    tensor in descending order (ties: the smaller column first), their softmax shares (fp32)
    and columns (int32), and the rows' log-sum-exp."""
    import torch

    if not isinstance(x, torch.Tensor) or not x.is_cuda or x.dtype != torch.float32:
        raise TypeError("x must be a CUDA fp32 tensor")
    if x.dim() != 2 or not x.is_contiguous():
        raise TypeError("x must be a contiguous [rows, cols] tensor")
    rows, cols = x.shape
    if values is None:
        values = torch.empty((rows, k), dtype=torch.float32, device=x.device)
    if indices is None:
        indices = torch.empty((rows, k), dtype=torch.int32, device=x.device)
    if lse is None and return_lse:
        lse = torch.empty((rows,), dtype=torch.float32, device=x.device)
    rc = osm_softmax_topk_raw(x.data_ptr(), rows, cols, k, values.data_ptr(), indices.data_ptr(),
                              lse.data_ptr() if lse is not None else None, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "osm_softmax_topk")
    return values, indices, lse


def fa_bwd(q, k, v, o, do, lse, scale=None, causal=False, workspace=None, stream=None):
    """(dQ, dK, dV) of fa_fwd's attention for the output gradient do (CUDA bf16 [B,H,N,d]),
    given the forward's o and lse.  `workspace` may be an fp32 CUDA tensor of B*H*N floats;
    otherwise it is allocated here (the library never allocates)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 [B, H, N, d] tensor")
        if t.shape != q.shape:
            raise ValueError("q, k, v, o, do must share one shape")
    B, H, N, d = q.shape
    if lse.dtype != torch.float32 or lse.shape != (B, H, N) or not lse.is_contiguous():
        raise TypeError("lse must be a contiguous fp32 [B, H, N] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(q), torch.empty_like(q)
    ws_d = (torch.empty(B * H * N, dtype=torch.float32, device=q.device) if workspace is None
            else workspace)
    rc = fa_bwd_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                    lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws_d.data_ptr(),
                    B, H, N, d, scale, causal, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def fa_bwd_gqa_raw(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr, ws_ptr,
                   B, H, H_kv, N, d, scale, causal, kv_lens_ptr, stream_ptr):
    return lib().fa_bwd_gqa(q_ptr, k_ptr, v_ptr, o_ptr, do_ptr, lse_ptr, dq_ptr, dk_ptr, dv_ptr,
                            ws_ptr, int(B), int(H), int(H_kv), int(N), int(d), float(scale),
                            int(bool(causal)), kv_lens_ptr, stream_ptr)


def fa_bwd_gqa(q, k, v, o, do, lse, kv_lens=None, scale=None, causal=False, workspace=None,
               stream=None):
    """(dQ, dK, dV) of fa_fwd_gqa's attention for the output gradient do: q, o, do CUDA bf16
    [B,H,N,d], k, v [B,H_kv,N,d], lse fp32 [B,H,N], optional kv_lens CUDA int32 [B].  dK, dV
    are [B,H_kv,N,d] (a shared key/value head's gradients sum over its query heads)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("do", do)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 [B, H, N, d] tensor")
    B, H, N, d = q.shape
    H_kv = k.shape[1]
    if o.shape != q.shape or do.shape != q.shape or k.shape != (B, H_kv, N, d) \
            or v.shape != k.shape:
        raise ValueError("q, o, do must be [B, H, N, d] and k, v [B, H_kv, N, d]")
    if lse.dtype != torch.float32 or lse.shape != (B, H, N) or not lse.is_contiguous():
        raise TypeError("lse must be a contiguous fp32 [B, H, N] tensor")
    if kv_lens is not None and (not isinstance(kv_lens, torch.Tensor) or not kv_lens.is_cuda
                                or kv_lens.dtype != torch.int32 or kv_lens.shape != (B,)):
        raise TypeError("kv_lens must be a CUDA int32 [B] tensor")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    ws_d = (torch.empty(B * H * N, dtype=torch.float32, device=q.device) if workspace is None
            else workspace)
    rc = fa_bwd_gqa_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), do.data_ptr(),
                        lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                        ws_d.data_ptr(), B, H, H_kv, N, d, scale, causal,
                        kv_lens.data_ptr() if kv_lens is not None else None,
                        _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_gqa")
    return dq, dk, dv


def fa_fwd_mask(q, k, v, mask_bits, scale=None, causal=False, out=None, lse=None, stream=None,
                skip_tiles=True, tile_map=None):
    """Attention of q [B,H,Nq,d] over k, v [B,H,Nk,d] (CUDA bf16) with an explicit mask:
    mask_bits is the CUDA uint32/int32 tensor [B or 1, H or 1, Nq, 4 * ceil(Nk / 128)] that
    inputs.pack_mask builds (size-1 leading dimensions repeat).  skip_tiles: pass a tile map
    (tile_map, a CUDA int32 tensor of at least mask_plan words, or one made here) so that key
    tiles with no allowed key are skipped.  Returns (O, LSE)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 [B, H, N, d] tensor")
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    if k.shape != (B, H, Nk, d) or v.shape != k.shape:
        raise ValueError("k, v must be [B, H, Nk, d] with q's B, H and d")
    W = 4 * ((Nk + 127) // 128)
    if (not isinstance(mask_bits, torch.Tensor) or not mask_bits.is_cuda
            or mask_bits.dtype not in (torch.int32, torch.uint32) or mask_bits.dim() != 4
            or not mask_bits.is_contiguous() or tuple(mask_bits.shape[2:]) != (Nq, W)
            or mask_bits.shape[0] not in (1, B) or mask_bits.shape[1] not in (1, H)):
        raise TypeError("mask_bits must be a contiguous CUDA int32 [B or 1, H or 1, Nq, W]")
    hs = Nq * W if mask_bits.shape[1] == H and H > 1 else 0
    bs = mask_bits.shape[1] * Nq * W if mask_bits.shape[0] == B and B > 1 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    O = torch.empty_like(q) if out is None else out
    L = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    tm_ptr, tm_words = 0, 0
    if skip_tiles:
        need = mask_plan(B, H, Nq, Nk, bs, hs)
        if tile_map is None:
            tile_map = torch.empty(max(need, 1), dtype=torch.int32, device=q.device)
        if (not isinstance(tile_map, torch.Tensor) or not tile_map.is_cuda
                or tile_map.dtype not in (torch.int32, torch.uint32)
                or not tile_map.is_contiguous() or tile_map.numel() < need):
            raise TypeError(f"tile_map must be a contiguous CUDA int32 tensor of >= {need} words")
        tm_ptr, tm_words = tile_map.data_ptr(), tile_map.numel()
    rc = fa_fwd_mask_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(), L.data_ptr(),
                         B, H, Nq, Nk, d, scale, causal, mask_bits.data_ptr(), bs, hs,
                         tm_ptr, tm_words, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_mask")
    return O, L


def fa_fwd_gqa_mask(q, k, v, mask_bits, kv_lens=None, n_splits=0, scale=None, causal=False,
                    out=None, lse=None, stream=None, skip_tiles=True, tile_map=None,
                    workspace=None):
    """Attention of q [B,H,Nq,d] over k, v [B,H_kv,Nk,d] (CUDA bf16, H_kv divides H) with an
    explicit mask (mask_bits as for fa_fwd_mask, over the H query heads), optional key lengths
    kv_lens (CUDA int32 [B]) and n_splits key ranges (0: chosen by the plan call; 1: one pass).
    skip_tiles / tile_map as for fa_fwd_mask; workspace: (ws_O, ws_LSE) fp32 CUDA tensors of
    at least the plan's sizes, or made here.  Returns (O, LSE)."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or not t.is_cuda:
            raise TypeError(f"{name} must be a CUDA tensor")
        if t.dtype != torch.bfloat16 or t.dim() != 4 or not t.is_contiguous():
            raise TypeError(f"{name} must be a contiguous bf16 [B, H, N, d] tensor")
    B, H, Nq, d = q.shape
    H_kv, Nk = k.shape[1], k.shape[2]
    if k.shape != (B, H_kv, Nk, d) or v.shape != k.shape:
        raise ValueError("k, v must be [B, H_kv, Nk, d] with q's B and d")
    W = 4 * ((Nk + 127) // 128)
    if (not isinstance(mask_bits, torch.Tensor) or not mask_bits.is_cuda
            or mask_bits.dtype not in (torch.int32, torch.uint32) or mask_bits.dim() != 4
            or not mask_bits.is_contiguous() or tuple(mask_bits.shape[2:]) != (Nq, W)
            or mask_bits.shape[0] not in (1, B) or mask_bits.shape[1] not in (1, H)):
        raise TypeError("mask_bits must be a contiguous CUDA int32 [B or 1, H or 1, Nq, W]")
    if kv_lens is not None and (not isinstance(kv_lens, torch.Tensor) or not kv_lens.is_cuda
                                or kv_lens.dtype != torch.int32 or kv_lens.shape != (B,)):
        raise TypeError("kv_lens must be a CUDA int32 [B] tensor")
    hs = Nq * W if mask_bits.shape[1] == H and H > 1 else 0
    bs = mask_bits.shape[1] * Nq * W if mask_bits.shape[0] == B and B > 1 else 0
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    splits, wo, wl, need = gqa_mask_plan(B, H, H_kv, Nq, Nk, d, bs, hs, n_splits)
    O = torch.empty_like(q) if out is None else out
    L = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    tm_ptr, tm_words = 0, 0
    if skip_tiles:
        if tile_map is None:
            tile_map = torch.empty(max(need, 1), dtype=torch.int32, device=q.device)
        if (not isinstance(tile_map, torch.Tensor) or not tile_map.is_cuda
                or tile_map.dtype not in (torch.int32, torch.uint32)
                or not tile_map.is_contiguous() or tile_map.numel() < need):
            raise TypeError(f"tile_map must be a contiguous CUDA int32 tensor of >= {need} words")
        tm_ptr, tm_words = tile_map.data_ptr(), tile_map.numel()
    ws_o = ws_l = None
    if splits > 1:
        if workspace is None:
            workspace = (torch.empty(wo, dtype=torch.float32, device=q.device),
                         torch.empty(wl, dtype=torch.float32, device=q.device))
        ws_o, ws_l = workspace
        if ws_o.numel() < wo or ws_l.numel() < wl:
            raise ValueError("workspace too small for the plan")
    rc = fa_fwd_gqa_mask_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), O.data_ptr(),
                             L.data_ptr(), B, H, H_kv, Nq, Nk, d, scale, causal,
                             kv_lens.data_ptr() if kv_lens is not None else None,
                             mask_bits.data_ptr(), bs, hs, tm_ptr, tm_words, max(splits, 1),
                             ws_o.data_ptr() if ws_o is not None else None,
                             ws_l.data_ptr() if ws_l is not None else None,
                             _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_gqa_mask")
    return O, L

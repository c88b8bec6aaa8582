"""Python binding of the bsattn C ABI (block-sparse attention for GB300 / sm_103a).

Argument marshalling only: every function passes tensor data pointers, shapes and the
current CUDA stream to the same-named C entry point of libbsattn.so and raises on a
non-zero status.  torch supplies device memory (outputs, workspaces) and streams; no step of
the computation runs in Python, and there is no CPU fallback: if the library is missing
the calls raise.

    bsattn_prefill(q, k, v, block_mask, is_causal)                      -> out
    bsattn_decode_varlen(q, k, v, cache_seqlens, block_indices, num_splits=0) -> out
    bsattn_mask_from_topk(scores, topk, use_dense_for_last_block, apply_tril)  -> mask
    bsattn_mask_from_threshold(scores, thr, use_dense_for_last_block, apply_tril) -> mask
    bsattn_num_splits_heuristic(...)                                     -> int
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

__all__ = [
    "BSATTN_OK", "BSATTN_ERR_INVALID_ARG", "BSATTN_ERR_UNSUPPORTED", "BSATTN_ERR_CUDA",
    "BSATTN_ERR_TIMEOUT", "BSATTN_ERR_BAD_INDEX", "BsattnError", "library_path", "load",
    "bsattn_prefill", "bsattn_prefill_bs", "bsattn_prefill_workspace_size", "bsattn_decode_varlen",
    "bsattn_decode_workspace_size", "bsattn_decode_default_splits", "bsattn_num_splits_heuristic",
    "bsattn_mask_from_topk", "bsattn_mask_from_threshold", "bsattn_get_device_status",
    "bsattn_set_wait_budget_ns", "bsattn_status_string", "bsattn_version", "workspace",
    "bsattn_decode_varlen_mask", "bsattn_decode_paged", "bsattn_mask_from_cumulative_threshold",
    "bsattn_decode_varlen_noalloc", "bsattn_decode_noalloc_status",
]

BSATTN_OK = 0
BSATTN_ERR_INVALID_ARG = 1
BSATTN_ERR_UNSUPPORTED = 2
BSATTN_ERR_CUDA = 4
BSATTN_ERR_TIMEOUT = 8
BSATTN_ERR_BAD_INDEX = 16

_F16, _BF16 = 0, 1
_lock = threading.Lock()
_lib = None


class BsattnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} failed: {bsattn_status_string(status)} ({status})")
        self.status = status


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads libbsattn.so (building it with nvcc first if it is missing)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                if not build_if_missing:
                    raise OSError(f"{path} is not built; run block_sparse_attention_gb300.build")
                _build.build()
            lib = ctypes.CDLL(path)
            P, I, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            sig = {
                "bsattn_status_string": ([I], ctypes.c_char_p),
                "bsattn_version": ([], ctypes.c_char_p),
                "bsattn_prefill": ([P, P, P, P, I, P, I, I, I, I, I, I, P, Z, P], I),
                "bsattn_prefill_bs": ([P, P, P, P, I, I, P, I, I, I, I, I, I, P, Z, P], I),
                "bsattn_prefill_workspace_size": ([I, I, I, I], Z),
                "bsattn_decode_varlen": ([P, P, P, P, P, I, P, I, I, I, I, I, I, I, P, Z, P], I),
                "bsattn_decode_workspace_size": ([I, I, I, I, I, I], Z),
                "bsattn_decode_default_splits": ([I, I, I, I, I], I),
                "bsattn_num_splits_heuristic": ([I, I, I, I, ctypes.c_longlong, I, I], I),
                "bsattn_mask_from_topk": ([P, I, I, I, I, I, I, I, P], I),
                "bsattn_mask_from_threshold": ([P, I, I, I, I, ctypes.c_float, I, I, P], I),
                "bsattn_get_device_status": ([P, P], I),
                "bsattn_decode_varlen_mask": ([P, P, P, P, P, I, P, I, I, I, I, I, I, I, P, Z, P], I),
                "bsattn_decode_paged": ([P, P, P, P, P, P, I, P, I, I, I, I, I, I, I, I, I, P, Z, P], I),
                "bsattn_mask_from_cumulative_threshold": ([P, I, I, I, I, ctypes.c_double, I, P], I),
                "bsattn_set_wait_budget_ns": ([ctypes.c_ulonglong], None),
                "bsattn_decode_varlen_noalloc": ([P, P, P, P, P, I, P, I, I, I, I, I, I, I, P], I),
                "bsattn_decode_noalloc_status": ([P], I),
            }
            for name, (args, res) in sig.items():
                f = getattr(lib, name)
                f.argtypes = args
                f.restype = res
            _lib = lib
    return _lib


def _check(fn: str, rc: int):
    if rc != BSATTN_OK:
        raise BsattnError(fn, rc)


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return _F16
    if t.dtype == torch.bfloat16:
        return _BF16
    raise TypeError(f"bsattn takes fp16 or bf16 tensors, got {t.dtype}")


def _cuda_contig(name: str, t: torch.Tensor) -> torch.Tensor:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


# zero-filled workspaces, one per (device, purpose); the kernels leave them zeroed
_ws_cache: dict = {}


def workspace(device, purpose: str, nbytes: int) -> torch.Tensor:
    """The zero-filled workspace this binding passes for `purpose` on `device`."""
    device = torch.device(device)
    if device.type == "cuda" and device.index is None:
        device = torch.device("cuda", torch.cuda.current_device())
    key = (device.index, purpose)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < nbytes:
        buf = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf


def bsattn_status_string(status: int) -> str:
    return load().bsattn_status_string(int(status)).decode()


def bsattn_version() -> str:
    return load().bsattn_version().decode()


def bsattn_prefill_workspace_size(B: int, H: int, Sq: int, Sk: int) -> int:
    return int(load().bsattn_prefill_workspace_size(B, H, Sq, Sk))


def bsattn_prefill(q, k, v, block_mask, is_causal: bool, out=None, ws=None, block_size: int = 64):
    """Block-sparse attention forward.  q [B,H,Sq,d], k/v [B,H,Sk,d] fp16|bf16 CUDA;
    block_mask [B,H,ceil(Sq/bs),ceil(Sk/bs)] uint8/bool CUDA, bs = block_size (64 or 128)."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("block_mask", block_mask)):
        _cuda_contig(name, t)
    B, H, Sq, d = q.shape
    Sk = k.shape[2]
    if block_mask.dtype == torch.bool:
        block_mask = block_mask.view(torch.uint8)
    if block_mask.dtype not in (torch.uint8, torch.int8):
        raise TypeError("block_mask must be uint8, int8 or bool")
    if tuple(block_mask.shape) != (B, H, -(-Sq // block_size), -(-Sk // block_size)):
        raise ValueError(f"block_mask shape {tuple(block_mask.shape)} does not match q/k")
    if k.shape != v.shape or k.shape[:2] != q.shape[:2] or k.shape[3] != d:
        raise ValueError("q, k, v shapes disagree")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(q.device, "prefill", bsattn_prefill_workspace_size(B, H, Sq, Sk))
    if block_size == 64:
        rc = lib.bsattn_prefill(q.data_ptr(), k.data_ptr(), v.data_ptr(), block_mask.data_ptr(),
                                int(bool(is_causal)), out.data_ptr(), B, H, Sq, Sk, d, _dtype_code(q),
                                ws.data_ptr(), ws.numel(), _stream(q.device))
    else:
        rc = lib.bsattn_prefill_bs(q.data_ptr(), k.data_ptr(), v.data_ptr(), block_mask.data_ptr(),
                                   int(block_size), int(bool(is_causal)), out.data_ptr(), B, H, Sq,
                                   Sk, d, _dtype_code(q), ws.data_ptr(), ws.numel(), _stream(q.device))
    _check("bsattn_prefill", rc)
    return out


def bsattn_decode_default_splits(B: int, Hkv: int, max_sel: int, d: int = 128,
                                 num_sms: int = 0) -> int:
    return int(load().bsattn_decode_default_splits(B, Hkv, max_sel, d, num_sms))


def bsattn_decode_workspace_size(B, Hq, Hkv, d, max_sel, num_splits=0) -> int:
    return int(load().bsattn_decode_workspace_size(B, Hq, Hkv, d, max_sel, num_splits))


def bsattn_decode_varlen(q, k, v, cache_seqlens, block_indices, num_splits: int = 0, out=None,
                         ws=None):
    """GQA varlen sparse decode.  q [B,Hq,d]; k/v [B,Smax,Hkv,d] fp16|bf16 CUDA;
    cache_seqlens int32 [B]; block_indices int32 [B,Hkv,max_sel] (-1 = empty)."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("cache_seqlens", cache_seqlens),
                    ("block_indices", block_indices)):
        _cuda_contig(name, t)
    if cache_seqlens.dtype != torch.int32 or block_indices.dtype != torch.int32:
        raise TypeError("cache_seqlens and block_indices must be int32")
    B, Hq, d = q.shape
    _, Smax, Hkv, _ = k.shape
    max_sel = block_indices.shape[2]
    if tuple(block_indices.shape[:2]) != (B, Hkv) or k.shape != v.shape:
        raise ValueError("decode shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(q.device, "decode",
                       bsattn_decode_workspace_size(B, Hq, Hkv, d, max_sel, num_splits))
    rc = lib.bsattn_decode_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                  cache_seqlens.data_ptr(), block_indices.data_ptr(),
                                  int(num_splits), out.data_ptr(), B, Hq, Hkv, Smax, d, max_sel,
                                  _dtype_code(q), ws.data_ptr(), ws.numel(), _stream(q.device))
    _check("bsattn_decode_varlen", rc)
    return out


def bsattn_decode_varlen_noalloc(q, k, v, cache_seqlens, block_indices, num_splits: int = 0, out=None):
    """bsattn_decode_varlen on the library's own fixed scratch array (no workspace argument, no
    device allocation by the library; `out` is allocated here when not given)."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("cache_seqlens", cache_seqlens),
                    ("block_indices", block_indices)):
        _cuda_contig(name, t)
    if cache_seqlens.dtype != torch.int32 or block_indices.dtype != torch.int32:
        raise TypeError("cache_seqlens and block_indices must be int32")
    B, Hq, d = q.shape
    _, Smax, Hkv, _ = k.shape
    max_sel = block_indices.shape[2]
    if tuple(block_indices.shape[:2]) != (B, Hkv) or k.shape != v.shape:
        raise ValueError("decode shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    rc = lib.bsattn_decode_varlen_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                          cache_seqlens.data_ptr(), block_indices.data_ptr(),
                                          int(num_splits), out.data_ptr(), B, Hq, Hkv, Smax, d,
                                          max_sel, _dtype_code(q), _stream(q.device))
    _check("bsattn_decode_varlen_noalloc", rc)
    return out


def bsattn_decode_noalloc_status(device=None) -> int:
    """Reads and clears the status word of the allocation-free decode on `device` (default: the
    current one); syncs that device's current stream."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    return int(load().bsattn_decode_noalloc_status(_stream(dev)))


def bsattn_decode_varlen_mask(q, k, v, cache_seqlens, block_mask, num_splits: int = 0, out=None,
                              ws=None):
    """GQA varlen sparse decode, block-mask form.  block_mask [B,Hkv,num_blocks] uint8/bool."""
    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("cache_seqlens", cache_seqlens),
                    ("block_mask", block_mask)):
        _cuda_contig(name, t)
    if block_mask.dtype == torch.bool:
        block_mask = block_mask.view(torch.uint8)
    if cache_seqlens.dtype != torch.int32 or block_mask.dtype != torch.uint8:
        raise TypeError("cache_seqlens must be int32 and block_mask uint8/bool")
    B, Hq, d = q.shape
    _, Smax, Hkv, _ = k.shape
    nb = block_mask.shape[2]
    if tuple(block_mask.shape[:2]) != (B, Hkv) or k.shape != v.shape:
        raise ValueError("decode shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(q.device, "decode", bsattn_decode_workspace_size(B, Hq, Hkv, d, nb, num_splits))
    rc = lib.bsattn_decode_varlen_mask(q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                       cache_seqlens.data_ptr(), block_mask.data_ptr(),
                                       int(num_splits), out.data_ptr(), B, Hq, Hkv, Smax, d, nb,
                                       _dtype_code(q), ws.data_ptr(), ws.numel(), _stream(q.device))
    _check("bsattn_decode_varlen_mask", rc)
    return out


def bsattn_decode_paged(q, k_pages, v_pages, cache_seqlens, block_indices, block_table,
                        num_splits: int = 0, out=None, ws=None):
    """GQA varlen sparse decode over a paged KV cache.  k_pages/v_pages
    [num_pages, page_size, Hkv, d]; block_table int32 [B, max_pages_per_seq]."""
    lib = load()
    for name, t in (("q", q), ("k_pages", k_pages), ("v_pages", v_pages),
                    ("cache_seqlens", cache_seqlens), ("block_indices", block_indices),
                    ("block_table", block_table)):
        _cuda_contig(name, t)
    if (cache_seqlens.dtype, block_indices.dtype, block_table.dtype) != (torch.int32,) * 3:
        raise TypeError("cache_seqlens, block_indices and block_table must be int32")
    B, Hq, d = q.shape
    num_pages, page_size, Hkv, _ = k_pages.shape
    max_sel = block_indices.shape[2]
    if k_pages.shape != v_pages.shape or tuple(block_indices.shape[:2]) != (B, Hkv):
        raise ValueError("paged decode shapes disagree")
    if out is None:
        out = torch.empty_like(q)
    if ws is None:
        ws = workspace(q.device, "decode", bsattn_decode_workspace_size(B, Hq, Hkv, d, max_sel, num_splits))
    rc = lib.bsattn_decode_paged(q.data_ptr(), k_pages.data_ptr(), v_pages.data_ptr(),
                                 cache_seqlens.data_ptr(), block_indices.data_ptr(),
                                 block_table.data_ptr(), int(num_splits), out.data_ptr(), B, Hq,
                                 Hkv, num_pages, page_size, block_table.shape[1], d, max_sel,
                                 _dtype_code(q), ws.data_ptr(), ws.numel(), _stream(q.device))
    _check("bsattn_decode_paged", rc)
    return out


def bsattn_mask_from_cumulative_threshold(attn_sum, threshold: float, causal: bool = True):
    """Host-side XAttention cumulative-threshold block mask; CPU uint8 tensor."""
    s = _host_scores(attn_sum)
    B, H, nq, nk = s.shape
    out = torch.empty(s.shape, dtype=torch.uint8)
    rc = load().bsattn_mask_from_cumulative_threshold(s.data_ptr(), B, H, nq, nk, float(threshold),
                                                      int(bool(causal)), out.data_ptr())
    _check("bsattn_mask_from_cumulative_threshold", rc)
    return out


def bsattn_num_splits_heuristic(total_mblocks, num_SMs, num_n_blocks, num_m_blocks,
                                size_one_kv_head, is_causal_or_local, max_splits) -> int:
    return int(load().bsattn_num_splits_heuristic(int(total_mblocks), int(num_SMs),
                                                  int(num_n_blocks), int(num_m_blocks),
                                                  int(size_one_kv_head),
                                                  int(bool(is_causal_or_local)), int(max_splits)))


def _host_scores(scores) -> torch.Tensor:
    s = torch.as_tensor(scores)
    if s.dim() != 4:
        raise ValueError("scores must be [B, H, nq, nk]")
    return s.detach().to("cpu", torch.float32).contiguous()


def bsattn_mask_from_topk(scores, topk: int, use_dense_for_last_block: bool = False,
                          apply_tril: bool = True) -> torch.Tensor:
    """Host-side top-k block mask; returns a CPU uint8 tensor of the scores' shape."""
    s = _host_scores(scores)
    B, H, nq, nk = s.shape
    out = torch.empty(s.shape, dtype=torch.uint8)
    rc = load().bsattn_mask_from_topk(s.data_ptr(), B, H, nq, nk, int(topk),
                                      int(bool(use_dense_for_last_block)), int(bool(apply_tril)),
                                      out.data_ptr())
    _check("bsattn_mask_from_topk", rc)
    return out


def bsattn_mask_from_threshold(scores, threshold: float, use_dense_for_last_block: bool = False,
                               apply_tril: bool = True) -> torch.Tensor:
    """Host-side threshold block mask (score > threshold); CPU uint8 tensor."""
    s = _host_scores(scores)
    B, H, nq, nk = s.shape
    out = torch.empty(s.shape, dtype=torch.uint8)
    rc = load().bsattn_mask_from_threshold(s.data_ptr(), B, H, nq, nk, float(threshold),
                                           int(bool(use_dense_for_last_block)),
                                           int(bool(apply_tril)), out.data_ptr())
    _check("bsattn_mask_from_threshold", rc)
    return out


def bsattn_get_device_status(ws: torch.Tensor) -> int:
    """Reads and clears the device status word of a workspace (syncs its stream)."""
    return int(load().bsattn_get_device_status(ws.data_ptr(), _stream(ws.device)))


def bsattn_set_wait_budget_ns(ns: int) -> None:
    load().bsattn_set_wait_budget_ns(int(ns))

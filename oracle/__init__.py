"""fp64 CPU oracle for block-sparse attention -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never calls it and
shares no code with it.

Contents, each a plain restatement of what the pages define:

* ``prefill`` / ``prefill_rows`` / ``decode_varlen`` / ``decode_paged``:
  ctypes wrappers over ``bsattn_oracle.c`` (fp64 masked softmax attention).
* ``mask_from_topk`` / ``mask_from_threshold``: the block-mask builders of the
  TileLang block-sparse Flash-Attention guide, sections 3.1 and 3.2.
* ``num_splits_heuristic``: the split-count rule of the same guide, section 6.3.
* ``decode_mask_to_indices``: the block-mask form of the decode input (guide,
  section 6) turned into the equivalent index set.
* ``find_blocks_chunked``: the cumulative-threshold block selection of the
  XAttention algorithm guide ("block selection algorithm" section).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bsattn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

F16, BF16, F64 = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (OpenMP) into oracle/_build/liboracle.so."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-Wall",
                        "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_double
            lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_f64.restype = D
            lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.oracle_bf16_to_f64.restype = D
            lib.oracle_num_threads.restype = I
            lib.oracle_prefill_rows.argtypes = [P, P, P, I, P, I, I, I, I, I, P, I, P]
            lib.oracle_prefill.argtypes = [P, P, P, I, P, I, I, I, I, I, I, I, P]
            lib.oracle_decode.argtypes = [P, P, P, I, P, P, I, I, I, I, I, I, I, P]
            lib.oracle_decode_paged.argtypes = [P, P, P, I, P, P, P, I, I, I, I, I, I, I, I, I, P]
            for f in (lib.oracle_prefill_rows, lib.oracle_prefill, lib.oracle_decode,
                      lib.oracle_decode_paged):
                f.restype = I
            _lib = lib
    return _lib


def num_threads() -> int:
    return _load().oracle_num_threads()


def _raw(x):
    """(contiguous numpy array of the raw storage, dtype code) for a tensor/array."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.float16:
                return x.view(torch.int16).numpy().view(np.uint16), F16
            if x.dtype == torch.bfloat16:
                return x.view(torch.int16).numpy().view(np.uint16), BF16
            if x.dtype == torch.float64:
                return x.numpy(), F64
            raise TypeError(f"oracle inputs must be fp16, bf16 or fp64, got {x.dtype}")
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(x)
    if a.dtype == np.float16:
        return a.view(np.uint16), F16
    if a.dtype == np.float64:
        return a, F64
    raise TypeError(f"oracle inputs must be fp16, bf16 or fp64, got {a.dtype}")


def _u8(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            return (x != 0).to(torch.uint8).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x) != 0, dtype=np.uint8)


def _i32(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return np.ascontiguousarray(x.detach().cpu().numpy().astype(np.int32))
    except ImportError:  # pragma: no cover
        pass
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def f16_to_f64(bits: int) -> float:
    return _load().oracle_f16_to_f64(bits)


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


# --------------------------------------------------------------------------- prefill

def prefill(q, k, v, block_mask, is_causal: bool, block: int = 64) -> np.ndarray:
    """Block-sparse attention forward, fp64.  q [B,H,Sq,d]; k,v [B,H,Sk,d];
    block_mask [B,H,ceil(Sq/block),ceil(Sk/block)] (nonzero = visit).
    Returns out [B,H,Sq,d] float64; rows with no visible key are exactly 0."""
    qa, dt = _raw(q)
    ka, dtk = _raw(k)
    va, dtv = _raw(v)
    assert dt == dtk == dtv, "q, k, v must share a dtype"
    B, H, Sq, d = qa.shape
    Sk = ka.shape[2]
    m = _u8(block_mask)
    nq, nk = -(-Sq // block), -(-Sk // block)
    assert m.shape == (B, H, nq, nk), (m.shape, (B, H, nq, nk))
    out = np.empty((B, H, Sq, d), np.float64)
    rc = _load().oracle_prefill(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(m), int(bool(is_causal)),
                                B, H, Sq, Sk, d, block, _ptr(out))
    if rc:
        raise ValueError("oracle_prefill rejected its arguments")
    return out


def prefill_rows(q, k, v, block_mask, is_causal: bool, b: int, h: int, rows, block: int = 64):
    """Selected query rows of one (batch, head); returns [len(rows), d] float64."""
    qa, dt = _raw(q[b, h])
    ka, _ = _raw(k[b, h])
    va, _ = _raw(v[b, h])
    Sq, d = qa.shape
    Sk = ka.shape[0]
    m = _u8(block_mask[b, h])
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int32))
    out = np.empty((len(r), d), np.float64)
    rc = _load().oracle_prefill_rows(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(m),
                                     int(bool(is_causal)), Sq, Sk, d, block, _ptr(r), len(r),
                                     _ptr(out))
    if rc:
        raise ValueError("oracle_prefill_rows rejected its arguments")
    return out


# --------------------------------------------------------------------------- decode

def decode_varlen(q, k, v, cache_seqlens, block_indices, block: int = 64) -> np.ndarray:
    """GQA varlen sparse decode, fp64.  q [B,Hq,d]; k,v [B,Smax,Hkv,d];
    cache_seqlens [B]; block_indices [B,Hkv,max_sel] (-1 = empty slot).
    Returns out [B,Hq,d] float64."""
    qa, dt = _raw(q)
    ka, _ = _raw(k)
    va, _ = _raw(v)
    B, Hq, d = qa.shape
    _, Smax, Hkv, _ = ka.shape
    sl = _i32(cache_seqlens)
    bi = _i32(block_indices)
    max_sel = bi.shape[2]
    out = np.empty((B, Hq, d), np.float64)
    rc = _load().oracle_decode(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(sl), _ptr(bi), B, Hq, Hkv,
                               Smax, d, max_sel, block, _ptr(out))
    if rc:
        raise ValueError("oracle_decode rejected its arguments")
    return out


def decode_paged(q, k_pages, v_pages, cache_seqlens, block_indices, block_table,
                 block: int = 64) -> np.ndarray:
    """Paged decode, fp64.  k_pages, v_pages [num_pages, page_size, Hkv, d];
    block_table [B, max_pages_per_seq]."""
    qa, dt = _raw(q)
    ka, _ = _raw(k_pages)
    va, _ = _raw(v_pages)
    B, Hq, d = qa.shape
    num_pages, page_size, Hkv, _ = ka.shape
    sl = _i32(cache_seqlens)
    bi = _i32(block_indices)
    bt = _i32(block_table)
    out = np.empty((B, Hq, d), np.float64)
    rc = _load().oracle_decode_paged(_ptr(qa), _ptr(ka), _ptr(va), dt, _ptr(sl), _ptr(bi),
                                     _ptr(bt), B, Hq, Hkv, num_pages, page_size, bt.shape[1], d,
                                     bi.shape[2], block, _ptr(out))
    if rc:
        raise ValueError("oracle_decode_paged rejected its arguments")
    return out


def decode_mask_to_indices(block_mask) -> np.ndarray:
    """Decode block-mask form [B,Hkv,num_blocks] -> the same set as an index table
    [B,Hkv,num_blocks], selected blocks in descending order, -1 padded."""
    m = _u8(block_mask)
    B, Hkv, nb = m.shape
    out = np.full((B, Hkv, nb), -1, np.int32)
    for b in range(B):
        for g in range(Hkv):
            sel = np.nonzero(m[b, g])[0][::-1]
            out[b, g, : len(sel)] = sel
    return out


# --------------------------------------------------------------------------- mask builders

def _scores(x) -> np.ndarray:
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().to(torch.float32).numpy()
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if a.ndim != 4:
        raise ValueError("scores must be [B, H, nq, nk]")
    if np.isnan(a).any():
        raise ValueError("scores contain NaN")
    return a


def _dense_last_then_tril(mask: np.ndarray, use_dense_for_last_block: bool, tril: bool):
    # Guide section 3.1: the last two query-block rows are forced all-True, then the
    # lower block triangle (column <= row) is kept.
    if use_dense_for_last_block:
        mask[:, :, -2:, :] = 1
    if tril:
        nq, nk = mask.shape[2:]
        keep = np.arange(nk)[None, :] <= np.arange(nq)[:, None]
        mask &= keep.astype(np.uint8)
    return mask


def mask_from_topk(scores, topk: int, use_dense_for_last_block: bool = False,
                   tril: bool = True) -> np.ndarray:
    """Guide section 3.1: per query-block row keep the `topk` highest-scoring key
    blocks.  Ties: the lower column index wins.  topk > nk keeps the whole row."""
    x = _scores(scores)
    if topk < 0:
        raise ValueError("topk must be >= 0")
    B, H, nq, nk = x.shape
    kk = min(int(topk), nk)
    rows = x.reshape(-1, nk)
    cols = np.broadcast_to(np.arange(nk), rows.shape)
    order = np.lexsort((cols, -rows), axis=-1)          # score descending, then column
    mask = np.zeros(rows.shape, np.uint8)
    np.put_along_axis(mask, order[:, :kk], 1, axis=-1)
    return _dense_last_then_tril(mask.reshape(B, H, nq, nk), use_dense_for_last_block, tril)


def mask_from_threshold(scores, threshold: float, use_dense_for_last_block: bool = False,
                        tril: bool = True) -> np.ndarray:
    """Guide section 3.2: keep the key blocks whose score exceeds the threshold."""
    x = _scores(scores)
    mask = (x > np.float32(threshold)).astype(np.uint8)
    return _dense_last_then_tril(mask, use_dense_for_last_block, tril)


# --------------------------------------------------------------------------- split count

def num_splits_heuristic(total_mblocks: int, num_SMs: int, num_n_blocks: int, num_m_blocks: int,
                         size_one_kv_head: int, is_causal_or_local: bool, max_splits: int) -> int:
    """Guide section 6.3: the smallest split count whose wave efficiency is within
    85% of the best, after the two early exits the section lists."""
    if total_mblocks >= 0.8 * num_SMs:
        size_l2 = 50 * 1024 * 1024
        if (size_one_kv_head > size_l2 and num_m_blocks > 2 * num_SMs
                and not is_causal_or_local):
            return min(math.ceil(size_one_kv_head / size_l2), max_splits)
        return 1
    if num_n_blocks <= 4:
        return 1
    limit = min(max_splits, num_SMs, num_n_blocks)
    eff = []
    for s in range(1, limit + 1):
        n_waves = total_mblocks * s / num_SMs
        eff.append(n_waves / math.ceil(n_waves))
    best = max(eff) if eff else 0.0
    for s in range(1, limit + 1):
        if eff[s - 1] >= 0.85 * best:
            return s
    return 1


def decode_num_splits(B: int, Hkv: int, max_sel: int, d: int, dv: int, num_SMs: int,
                      block: int = 64) -> int:
    """The guide's decode call of the heuristic: one m-block per (batch, kv head),
    the selected-block count as n-blocks, causal/local set, at most 128 splits."""
    size_one_kv_head = max_sel * block * (d + dv) * 2
    return num_splits_heuristic(B * Hkv, num_SMs, max_sel, 1, size_one_kv_head, True, 128)


# --------------------------------------------------------------------------- XAttention rule

def cumulative_pick(values, required: float):
    """The cumulative step of the XAttention block selection: visit the candidates
    from the largest weight down (ties: lower index first) and take each one while the
    sum of those already taken is still below `required`; so the candidate whose
    addition reaches `required` is taken too (the guide's worked example takes it).
    `values` maps candidate index -> weight.  Returns the taken indices in order."""
    order = sorted(values, key=lambda j: (-values[j], j))
    taken, acc = [], 0.0
    for j in order:
        if acc >= required:
            break
        taken.append(j)
        acc += values[j]
    return taken


def find_blocks_chunked(attn_sum, threshold: float, causal: bool = True) -> np.ndarray:
    """XAttention guide, block selection: per query block, keep the sink block
    (column 0) and, when causal, the diagonal block; then take the remaining blocks
    by ``cumulative_pick`` with required = threshold * (row total).
    Returns uint8 [B,H,nq,nk]."""
    x = np.asarray(attn_sum, dtype=np.float64)
    B, H, nq, nk = x.shape
    mask = np.zeros(x.shape, np.uint8)
    for b in range(B):
        for h in range(H):
            for i in range(nq):
                row = x[b, h, i]
                mask[b, h, i, 0] = 1
                if causal and i < nk:
                    mask[b, h, i, i] = 1
                total = 0.0
                for val in row:                  # the row total, summed left to right
                    total += float(val)
                rest = {j: float(row[j]) for j in range(nk) if not mask[b, h, i, j]}
                for j in cumulative_pick(rest, total * threshold):
                    mask[b, h, i, j] = 1
    return mask

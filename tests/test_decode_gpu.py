"""GPU parity of bsattn_decode_varlen (through the C ABI) against the fp64 oracle.

Tolerance: max |err| <= 2e-2 for bf16 inputs, <= 1e-2 for fp16.  Index handling is exact:
results must not depend on the order of the indices or on num_splits beyond rounding, a
selection with no blocks gives exactly 0, tokens past cache_seqlens are never used (they
hold NaN here), and an index past the sequence end is skipped and flagged.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

TOL = {torch.float16: 1e-2, torch.bfloat16: 2e-2}


@pytest.fixture(scope="module")
def bsa():
    import block_sparse_attention_gb300 as m
    m.load()
    return m


def _run(bsa, q, k, v, sl, idx, ns=0):
    dev = torch.device("cuda")
    out = bsa.bsattn_decode_varlen(q.to(dev), k.to(dev), v.to(dev), sl.to(dev),
                                   idx.to(dev), ns)
    torch.cuda.synchronize()
    return out.cpu()


def _err(got, want):
    return float(np.abs(got.double().numpy() - want).max())


def _small_case(Hq=8, Hkv=2, d=128, dtype=torch.bfloat16, fill=float("nan")):
    g = torch.Generator().manual_seed(Hq * 7 + d)
    B, Smax = 3, 700
    sl = torch.tensor([700, 1, 333], dtype=torch.int32)
    q = torch.randn(B, Hq, d, generator=g).to(dtype)
    k = torch.randn(B, Smax, Hkv, d, generator=g).to(dtype)
    v = torch.randn(B, Smax, Hkv, d, generator=g).to(dtype)
    for b in range(B):
        k[b, sl[b]:] = fill
        v[b, sl[b]:] = fill
    idx = torch.full((B, Hkv, 6), -1, dtype=torch.int32)
    idx[0, 0, :4] = torch.tensor([10, 7, 3, 0])
    idx[0, -1, :3] = torch.tensor([2, 9, 5])
    idx[1, 0, :1] = 0
    idx[2, 0, :2] = torch.tensor([5, 1])
    idx[2, -1, :6] = torch.tensor([0, 1, 2, 3, 4, 5])
    return q, k, v, sl, idx


@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (8, 1), (16, 8), (6, 3)])
@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float16),
                                     (64, torch.bfloat16), (128, torch.float16)])
@pytest.mark.parametrize("ns", [1, 2, 3, 6])
def test_decode_small_cases(bsa, Hq, Hkv, d, dtype, ns):
    q, k, v, sl, idx = _small_case(Hq, Hkv, d, dtype)
    got = _run(bsa, q, k, v, sl, idx, ns)
    want = oracle.decode_varlen(q, k, v, sl, idx)
    assert _err(got, want) <= TOL[dtype]
    zero = np.all(want == 0.0, axis=-1)          # heads whose selection is empty
    assert np.all(got.double().numpy()[zero] == 0.0)
    if Hkv > 1:
        assert zero.any()


def test_decode_bad_index_is_skipped_and_flagged(bsa):
    q, k, v, sl, idx = _small_case()
    idx[2, 0, 2] = 6            # seqlen 333 -> blocks 0..5 valid; 6 is past the end
    dev = torch.device("cuda")
    ws = bsa.workspace(dev, "decode", bsa.bsattn_decode_workspace_size(3, 8, 2, 128, 6, 2))
    bsa.bsattn_get_device_status(ws)
    got = _run(bsa, q, k, v, sl, idx, 2)
    assert bsa.bsattn_get_device_status(ws) & bsa.BSATTN_ERR_BAD_INDEX
    want = oracle.decode_varlen(q, k, v, sl, idx)
    assert _err(got, want) <= TOL[torch.bfloat16]


def _poison_unselected(k, v, sl, idx):
    """NaN in every valid token of a block that (b, kv head) does not select; the tokens
    past cache_seqlens keep what they hold."""
    B, Smax, Hkv, _ = k.shape
    nb = (Smax + 63) // 64
    sel = torch.zeros(B, Hkv, nb + 1, dtype=torch.bool)
    ids = idx.long().clamp(min=-1)
    sel.scatter_(2, torch.where(ids < 0, torch.full_like(ids, nb), ids), True)
    tok = torch.arange(Smax)
    valid = tok[None, :] < sl.long()[:, None]                        # [B, Smax]
    chosen = sel[:, :, tok // 64].permute(0, 2, 1)                   # [B, Smax, Hkv]
    poison = valid[:, :, None] & ~chosen
    kp, vp = k.clone(), v.clone()
    kp[poison] = float("nan")
    vp[poison] = float("nan")
    return kp, vp


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float16)])
@pytest.mark.parametrize("ns", [1, 3])
def test_decode_unselected_blocks_are_never_loaded(bsa, d, dtype, ns):
    """Valid blocks that a (b, kv head) does not select hold NaN (so do the tokens past
    cache_seqlens): the output matches the oracle on the clean cache bit for bit against the
    clean run -- the selection decides which tiles are read, not only which are used."""
    q, k, v, sl, idx = _small_case(8, 2, d, dtype)
    kp, vp = _poison_unselected(k, v, sl, idx)
    got = _run(bsa, q, kp, vp, sl, idx, ns)
    assert torch.equal(got, _run(bsa, q, k, v, sl, idx, ns))
    assert _err(got, oracle.decode_varlen(q, k, v, sl, idx)) <= TOL[dtype]


@pytest.fixture(scope="module")
def c5():
    cfg = synthetic.DECODE_CONFIGS["C5"]
    q, k, v, sl, idx = synthetic.decode_inputs(cfg, fill=float("nan"))
    want = oracle.decode_varlen(q, k, v, sl, idx)
    return cfg, q, k, v, sl, idx, want


@pytest.mark.parametrize("ns", [0, 1, 7, 19, 64])
def test_c5_full_size(bsa, c5, ns):
    cfg, q, k, v, sl, idx, want = c5
    got = _run(bsa, q, k, v, sl, idx, ns)
    assert _err(got, want) <= TOL[cfg.dtype]


@pytest.mark.parametrize("order", ["ascending", "shuffled"])
def test_c5_index_order_does_not_matter(bsa, c5, order):
    cfg, q, k, v, sl, idx, want = c5
    if order == "ascending":
        idx2 = idx.sort(dim=-1).values.contiguous()     # any -1 padding moves to the front
    else:
        g = torch.Generator().manual_seed(5)
        perm = torch.randperm(idx.shape[-1], generator=g)
        idx2 = idx[..., perm].contiguous()
    got = _run(bsa, q, k, v, sl, idx2, 0)
    assert _err(got, want) <= TOL[cfg.dtype]


def test_decode_empty_selection_is_zero(bsa, c5):
    cfg, q, k, v, sl, idx, _ = c5
    idx2 = idx.clone()
    idx2[3] = -1
    got = _run(bsa, q, k, v, sl, idx2, 0)
    assert torch.count_nonzero(got[3]) == 0
    want = oracle.decode_varlen(q, k, v, sl, idx2)
    assert _err(got, want) <= TOL[cfg.dtype]


def test_c5_unselected_blocks_are_never_loaded(bsa, c5):
    """C5 at full size with NaN in every valid token of every unselected block."""
    cfg, q, k, v, sl, idx, want = c5
    kp, vp = _poison_unselected(k, v, sl, idx)
    got = _run(bsa, q, kp, vp, sl, idx, 0)
    assert _err(got, want) <= TOL[cfg.dtype]
    assert torch.equal(got, _run(bsa, q, k, v, sl, idx, 0))


def test_decode_is_deterministic(bsa, c5):
    cfg, q, k, v, sl, idx, _ = c5
    assert torch.equal(_run(bsa, q, k, v, sl, idx, 0), _run(bsa, q, k, v, sl, idx, 0))


def test_decode_timeout_path_reports_and_recovers(bsa, c5):
    cfg, q, k, v, sl, idx, want = c5
    dev = torch.device("cuda")
    ns = 7
    ws = torch.zeros(bsa.bsattn_decode_workspace_size(8, 32, 8, 128, 64, ns), dtype=torch.uint8,
                     device=dev)
    args = (q.to(dev), k.to(dev), v.to(dev), sl.to(dev), idx.to(dev), ns)
    try:
        bsa.bsattn_set_wait_budget_ns(0)
        bsa.bsattn_decode_varlen(*args, ws=ws)
        torch.cuda.synchronize()
    finally:
        bsa.bsattn_set_wait_budget_ns(2_000_000_000)
    assert bsa.bsattn_get_device_status(ws) & bsa.BSATTN_ERR_TIMEOUT
    ws.zero_()
    got = bsa.bsattn_decode_varlen(*args, ws=ws).cpu()
    assert bsa.bsattn_get_device_status(ws) == 0
    assert _err(got, want) <= TOL[cfg.dtype]


# ----------------------------------------------------------------- block-mask and paged forms

def _mask_of(idx, nb):
    B, Hkv, _ = idx.shape
    m = torch.zeros(B, Hkv, nb, dtype=torch.uint8)
    for b in range(B):
        for g in range(Hkv):
            for t in idx[b, g].tolist():
                if t >= 0:
                    m[b, g, t] = 1
    return m


@pytest.mark.parametrize("ns", [0, 1, 3])
def test_decode_mask_form(bsa, ns):
    q, k, v, sl, idx = _small_case()
    nb = 11
    m = _mask_of(idx, nb)
    m[2, 0, 9] = 1                    # past seqlen 333 (6 blocks): selects no tokens
    dev = torch.device("cuda")
    got = bsa.bsattn_decode_varlen_mask(q.to(dev), k.to(dev), v.to(dev), sl.to(dev), m.to(dev), ns).cpu()
    want = oracle.decode_varlen(q, k, v, sl, oracle.decode_mask_to_indices(m))
    assert _err(got, want) <= TOL[torch.bfloat16]
    assert torch.equal(got, bsa.bsattn_decode_varlen_mask(q.to(dev), k.to(dev), v.to(dev), sl.to(dev),
                                                          m.to(dev), ns).cpu())


def test_c5_mask_form_matches_index_form(bsa, c5):
    cfg, q, k, v, sl, idx, want = c5
    m = _mask_of(idx, cfg.Smax // 64)
    dev = torch.device("cuda")
    got = bsa.bsattn_decode_varlen_mask(q.to(dev), k.to(dev), v.to(dev), sl.to(dev), m.to(dev), 16).cpu()
    assert _err(got, want) <= TOL[cfg.dtype]


def _paged(k, v, page, seed=1, extra=5):
    B, Smax, Hkv, d = k.shape
    per_seq = -(-Smax // page)
    num_pages = B * per_seq + extra
    g = torch.Generator().manual_seed(seed)
    table = torch.randperm(num_pages, generator=g)[: B * per_seq].reshape(B, per_seq).to(torch.int32)
    kp = torch.full((num_pages, page, Hkv, d), float("nan"), dtype=k.dtype)
    vp = torch.full_like(kp, float("nan"))
    for b in range(B):
        for pg in range(per_seq):
            seg = slice(pg * page, min((pg + 1) * page, Smax))
            n = seg.stop - seg.start
            kp[table[b, pg], :n] = k[b, seg]
            vp[table[b, pg], :n] = v[b, seg]
    return kp, vp, table


@pytest.mark.parametrize("page", [64, 128, 256])
@pytest.mark.parametrize("ns", [1, 3])
def test_decode_paged(bsa, page, ns):
    q, k, v, sl, idx = _small_case()
    kp, vp, table = _paged(k, v, page)
    dev = torch.device("cuda")
    got = bsa.bsattn_decode_paged(q.to(dev), kp.to(dev), vp.to(dev), sl.to(dev), idx.to(dev),
                                  table.to(dev), ns).cpu()
    want = oracle.decode_paged(q, kp, vp, sl, idx, table)
    assert _err(got, want) <= TOL[torch.bfloat16]
    contiguous = _run(bsa, q, k, v, sl, idx, ns)
    assert torch.equal(got, contiguous)        # same tiles, same order: same bits


def test_decode_paged_unmapped_page_is_flagged(bsa):
    q, k, v, sl, idx = _small_case()
    kp, vp, table = _paged(k, v, 128)
    table[2, 1] = -1                           # seq 2 blocks 2-3 lose their page
    dev = torch.device("cuda")
    ws = bsa.workspace(dev, "decode", bsa.bsattn_decode_workspace_size(3, 8, 2, 128, 6, 2))
    bsa.bsattn_get_device_status(ws)
    got = bsa.bsattn_decode_paged(q.to(dev), kp.to(dev), vp.to(dev), sl.to(dev), idx.to(dev),
                                  table.to(dev), 2).cpu()
    assert bsa.bsattn_get_device_status(ws) & bsa.BSATTN_ERR_BAD_INDEX
    # the oracle with those blocks removed
    idx2 = idx.clone()
    for gg in range(2):
        idx2[2, gg] = torch.where((idx2[2, gg] == 2) | (idx2[2, gg] == 3), torch.tensor(-1, dtype=torch.int32), idx2[2, gg])
    assert _err(got, oracle.decode_varlen(q, k, v, sl, idx2)) <= TOL[torch.bfloat16]

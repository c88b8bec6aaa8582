"""Pins for the fp64 oracle, against things other than the oracle itself.

Each test checks the oracle against a value the pages or mathematics fix:
library routines for the special cases they cover (torch's scaled-dot-product
attention in fp64 with a boolean mask built the way the TileLang block-sparse
guide's section 5 builds it, numpy's / torch's float widening, torch.topk),
closed forms (one visible key, zero query, two keys), invariants (masked K/V
never matter, index order never matters) and hand-worked examples under
tests/golden/.  A plausible slip in the oracle (wrong scale, transposed mask,
swapped K/V, off-by-one causal edge, wrong GQA head map, tail handling) fails
at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
import synthetic

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------- widening

def test_f16_widening_all_bit_patterns(oracle_mod):
    bits = np.arange(65536, dtype=np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.f16_to_f64(int(b)) for b in bits])
    assert np.array_equal(got, want, equal_nan=True)


def test_bf16_widening_all_bit_patterns(oracle_mod):
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16)
    want = bits.view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle_mod.bf16_to_f64(int(b) & 0xFFFF) for b in bits.tolist()])
    assert np.array_equal(got, want, equal_nan=True)


# ----------------------------------------------------------------- prefill vs library

def _token_mask(block_mask, Sq, Sk, causal, block=64):
    """Guide section 5: kron(block_mask, ones(block, block)), cropped, AND causal."""
    bm = torch.as_tensor(np.asarray(block_mask)).to(torch.float64)
    full = torch.kron(bm, torch.ones(block, block, dtype=torch.float64))[..., :Sq, :Sk] > 0
    if causal:
        # bottom-right aligned lower triangle (identical to tril when Sq == Sk)
        full = full & torch.ones(Sq, Sk, dtype=torch.bool).tril(diagonal=Sk - Sq)
    return full


def _sdpa(q, k, v, token_mask):
    return F.scaled_dot_product_attention(q.double(), k.double(), v.double(),
                                          attn_mask=token_mask)


def _check_vs_sdpa(q, k, v, block_mask, causal, tol=1e-12):
    Sq, Sk = q.shape[2], k.shape[2]
    tm = _token_mask(block_mask, Sq, Sk, causal)
    got = oracle.prefill(q, k, v, block_mask, causal)
    empty = ~tm.any(-1).numpy()
    assert np.all(got[empty] == 0.0), "rows with no visible key must be exactly 0"
    if (~empty).any():
        want = _sdpa(q, k, v, tm).numpy()
        err = np.abs(got[~empty] - want[~empty]).max()
        assert err <= tol, err


@pytest.mark.parametrize("S", [1, 63, 64, 65, 130])
@pytest.mark.parametrize("d", [1, 8, 64])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_brute_force_tiny_f64(S, d, causal):
    g = torch.Generator().manual_seed(S * 100 + d)
    q, k, v = (torch.randn(1, 1, S, d, generator=g, dtype=torch.float64) for _ in range(3))
    nb = math.ceil(S / 64)
    bm = (torch.rand(1, 1, nb, nb, generator=g) < 0.6).to(torch.uint8)
    _check_vs_sdpa(q, k, v, bm, causal)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_brute_force_multihead_halfprec(dtype, causal):
    # B=2, H=3 with an asymmetric random mask: catches (b,h) strides and a transposed mask
    q, k, v = synthetic.qkv(2, 3, 200, 200, 16, dtype, seed=3)
    bm = synthetic.random_block_mask(2, 3, 4, 4, 0.5, seed=3)
    _check_vs_sdpa(q, k, v, bm, causal)


@pytest.mark.parametrize("Sq,Sk", [(1, 130), (64, 200), (65, 129), (100, 100)])
def test_prefill_bottom_right_causal(Sq, Sk):
    g = torch.Generator().manual_seed(Sq + Sk)
    q = torch.randn(1, 2, Sq, 8, generator=g, dtype=torch.float64)
    k = torch.randn(1, 2, Sk, 8, generator=g, dtype=torch.float64)
    v = torch.randn(1, 2, Sk, 8, generator=g, dtype=torch.float64)
    bm = (torch.rand(1, 2, math.ceil(Sq / 64), math.ceil(Sk / 64), generator=g) < 0.7)
    _check_vs_sdpa(q, k, v, bm.to(torch.uint8), True)


@pytest.mark.parametrize("causal", [False, True])
def test_all_true_mask_is_dense_attention(causal):
    q, k, v = synthetic.qkv(1, 2, 300, 300, 32, torch.float64, seed=5)
    bm = torch.ones(1, 2, 5, 5, dtype=torch.uint8)
    got = oracle.prefill(q, k, v, bm, causal)
    want = F.scaled_dot_product_attention(q, k, v, is_causal=causal).numpy()
    assert np.abs(got - want).max() <= 1e-12


# ----------------------------------------------------------------- closed forms / invariants

def test_masked_blocks_never_change_output():
    q, k, v = synthetic.qkv(1, 2, 256, 256, 16, torch.float16, seed=11)
    bm = synthetic.random_block_mask(1, 2, 4, 4, 0.5, seed=11)
    base = oracle.prefill(q, k, v, bm, True)
    k2, v2 = k.clone(), v.clone()
    for h in range(2):
        for kb in range(4):
            # a key block matters only if some query block selects it at/below the diagonal
            used = any(bm[0, h, qb, kb] and kb <= qb for qb in range(4))
            if not used:
                k2[0, h, kb * 64:(kb + 1) * 64] = 7.0
                v2[0, h, kb * 64:(kb + 1) * 64] = -3.0
    got = oracle.prefill(q, k2, v2, bm, True)
    assert np.array_equal(got, base)


def test_causal_ignores_mask_entries_above_the_diagonal():
    q, k, v = synthetic.qkv(1, 2, 256, 256, 16, torch.bfloat16, seed=12)
    bm = synthetic.random_block_mask(1, 2, 4, 4, 0.5, seed=12)
    upper = bm | torch.ones(4, 4, dtype=torch.uint8).triu(1)
    assert np.array_equal(oracle.prefill(q, k, v, upper, True),
                          oracle.prefill(q, k, v, bm, True))


def test_single_visible_key_returns_its_value():
    # Sk = 129: the last key block holds exactly one key (j = 128); select only it.
    q, k, v = synthetic.qkv(1, 1, 129, 129, 8, torch.float64, seed=2)
    bm = torch.zeros(1, 1, 3, 3, dtype=torch.uint8)
    bm[..., 2] = 1
    got = oracle.prefill(q, k, v, bm, False)
    assert np.array_equal(got[0, 0], np.broadcast_to(v[0, 0, 128].numpy(), (129, 8)))
    # causal, diagonal block only: the first row of each query block sees one key
    bm = torch.eye(3, dtype=torch.uint8)[None, None]
    got = oracle.prefill(q, k, v, bm, True)
    for qb in range(3):
        i = qb * 64
        assert np.array_equal(got[0, 0, i], v[0, 0, i].numpy())


def test_zero_query_is_mean_of_visible_values():
    q, k, v = synthetic.qkv(1, 1, 192, 192, 16, torch.float64, seed=4)
    q = torch.zeros_like(q)
    bm = torch.tensor([[[[1, 0, 0], [0, 1, 0], [1, 0, 1]]]], dtype=torch.uint8)
    got = oracle.prefill(q, k, v, bm, True)
    vv = v[0, 0].numpy()
    for i in (0, 63, 64, 100, 128, 191):
        qb = i // 64
        vis = [j for j in range(192) if bm[0, 0, qb, j // 64] and j <= i]
        assert np.allclose(got[0, 0, i], vv[vis].mean(0), rtol=0, atol=1e-14)


def test_two_keys_closed_form_scale():
    # q = a*e0, k0 = e0, k1 = 0  ->  s0 = a/sqrt(d), s1 = 0
    d, a = 16, 3.0
    q = torch.zeros(1, 1, 1, d, dtype=torch.float64)
    q[..., 0] = a
    k = torch.zeros(1, 1, 2, d, dtype=torch.float64)
    k[0, 0, 0, 0] = 1.0
    v = torch.zeros(1, 1, 2, d, dtype=torch.float64)
    v[0, 0, 0, 0] = 1.0
    v[0, 0, 1, 1] = 1.0
    got = oracle.prefill(q, k, v, torch.ones(1, 1, 1, 1, dtype=torch.uint8), False)
    w0 = math.exp(a / math.sqrt(d))
    assert got[0, 0, 0, 0] == pytest.approx(w0 / (w0 + 1), abs=1e-15)
    assert got[0, 0, 0, 1] == pytest.approx(1 / (w0 + 1), abs=1e-15)


def test_empty_rows_are_exactly_zero():
    q, k, v = synthetic.qkv(1, 1, 130, 130, 8, torch.float16, seed=9)
    bm = torch.zeros(1, 1, 3, 3, dtype=torch.uint8)
    bm[0, 0, 1, 0] = 1
    got = oracle.prefill(q, k, v, bm, True)
    assert np.all(got[0, 0, :64] == 0.0) and np.all(got[0, 0, 128:] == 0.0)
    assert np.all(np.abs(got[0, 0, 64:128]).sum(-1) > 0)


def test_prefill_rows_matches_full():
    q, k, v = synthetic.qkv(2, 2, 150, 150, 8, torch.bfloat16, seed=6)
    bm = synthetic.random_block_mask(2, 2, 3, 3, 0.6, seed=6)
    full = oracle.prefill(q, k, v, bm, True)
    rows = [0, 5, 63, 64, 149]
    got = oracle.prefill_rows(q, k, v, bm, True, 1, 1, rows)
    assert np.array_equal(got, full[1, 1, rows])


# ----------------------------------------------------------------- decode

def _decode_case(B=3, Hq=8, Hkv=2, d=16, Smax=700, seed=0, fill=0.0):
    g = torch.Generator().manual_seed(seed)
    seqlens = torch.tensor([700, 1, 333][:B], dtype=torch.int32)
    q = torch.randn(B, Hq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, Smax, Hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, Smax, Hkv, d, generator=g).to(torch.bfloat16)
    for b in range(B):
        k[b, seqlens[b]:] = fill
        v[b, seqlens[b]:] = fill
    idx = torch.full((B, Hkv, 6), -1, dtype=torch.int32)
    idx[0, 0, :4] = torch.tensor([10, 7, 3, 0])
    idx[0, 1, :3] = torch.tensor([2, 9, 5])
    idx[1, 0, :1] = 0
    idx[2, 0, :2] = torch.tensor([5, 1])
    idx[2, 1, :6] = torch.tensor([0, 1, 2, 3, 4, 5])
    return q, k, v, seqlens, idx


def _decode_sdpa(q, k, v, seqlens, idx, block=64):
    B, Hq, d = q.shape
    Hkv = k.shape[2]
    out = np.zeros((B, Hq, d))
    for b in range(B):
        for h in range(Hq):
            gg = h // (Hq // Hkv)
            toks = sorted({p for t in idx[b, gg].tolist() if t >= 0
                           for p in range(t * block, min(t * block + block, int(seqlens[b])))})
            if not toks:
                continue
            kk = k[b, toks, gg].double()[None]
            vv = v[b, toks, gg].double()[None]
            out[b, h] = F.scaled_dot_product_attention(q[b, h].double()[None, None], kk[None],
                                                       vv[None])[0, 0, 0].numpy()
    return out


def test_decode_vs_sdpa_on_selected_tokens():
    q, k, v, sl, idx = _decode_case()
    got = oracle.decode_varlen(q, k, v, sl, idx)
    want = _decode_sdpa(q, k, v, sl, idx)
    assert np.abs(got - want).max() <= 1e-12
    # batch 1 (seqlen 1) selects block 0 -> one key -> its value exactly
    assert np.array_equal(got[1, :4], np.broadcast_to(v[1, 0, 0].double().numpy(), (4, 16)))
    # kv head 1 of batch 1 selects nothing -> exactly 0
    assert np.all(got[1, 4:] == 0.0)


def test_decode_all_blocks_is_dense_prefix_attention():
    q, k, v, sl, _ = _decode_case()
    nb = 11
    idx = torch.arange(nb, dtype=torch.int32).flip(0).expand(3, 2, nb).contiguous()
    got = oracle.decode_varlen(q, k, v, sl, idx)
    for b in range(3):
        n = int(sl[b])
        for h in range(8):
            gg = h // 4
            want = F.scaled_dot_product_attention(q[b, h].double()[None, None, None],
                                                  k[b, :n, gg].double()[None, None],
                                                  v[b, :n, gg].double()[None, None])
            assert np.abs(got[b, h] - want[0, 0, 0].numpy()).max() <= 1e-12


def test_decode_index_order_and_repeats_do_not_matter():
    q, k, v, sl, idx = _decode_case()
    base = oracle.decode_varlen(q, k, v, sl, idx)
    perm = idx.clone()
    perm[0, 0, :4] = torch.tensor([0, 3, 10, 7])
    perm[0, 1, :4] = torch.tensor([9, 9, 2, 5])      # a repeat
    assert np.array_equal(oracle.decode_varlen(q, k, v, sl, perm), base)


def test_decode_never_reads_past_seqlen():
    q, k, v, sl, idx = _decode_case(fill=float("nan"))
    got = oracle.decode_varlen(q, k, v, sl, idx)
    assert np.isfinite(got).all()
    q0, k0, v0, _, _ = _decode_case(fill=0.0)
    assert np.array_equal(got, oracle.decode_varlen(q0, k0, v0, sl, idx))


def test_decode_paged_matches_contiguous():
    q, k, v, sl, idx = _decode_case()
    B, Smax, Hkv, d = k.shape
    page = 128
    per_seq = math.ceil(Smax / page)
    num_pages = B * per_seq + 3
    g = torch.Generator().manual_seed(1)
    phys = torch.randperm(num_pages, generator=g)[: B * per_seq].reshape(B, per_seq).to(torch.int32)
    kp = torch.zeros(num_pages, page, Hkv, d, dtype=k.dtype)
    vp = torch.zeros_like(kp)
    for b in range(B):
        for p in range(per_seq):
            seg = slice(p * page, min((p + 1) * page, Smax))
            n = seg.stop - seg.start
            kp[phys[b, p], :n] = k[b, seg]
            vp[phys[b, p], :n] = v[b, seg]
    got = oracle.decode_paged(q, kp, vp, sl, idx, phys)
    assert np.array_equal(got, oracle.decode_varlen(q, k, v, sl, idx))


def test_decode_mask_form_equals_index_form():
    q, k, v, sl, idx = _decode_case()
    nb = 11
    m = torch.zeros(3, 2, nb, dtype=torch.uint8)
    for b in range(3):
        for gg in range(2):
            for t in idx[b, gg].tolist():
                if t >= 0:
                    m[b, gg, t] = 1
    conv = oracle.decode_mask_to_indices(m)
    assert np.array_equal(oracle.decode_varlen(q, k, v, sl, conv),
                          oracle.decode_varlen(q, k, v, sl, idx))


# ----------------------------------------------------------------- mask builders

def test_mask_builders_hand_worked_examples():
    spec = json.load(open(os.path.join(GOLDEN, "mask_builders_4x4.json")))
    scores = np.array(spec["scores"], np.float32)
    for c in spec["cases"]:
        fn = oracle.mask_from_topk if c["rule"] == "topk" else oracle.mask_from_threshold
        got = fn(scores, c["param"], c["dense_last"], c["tril"])
        assert np.array_equal(got[0, 0], np.array(c["expect"], np.uint8)), c["why"]


def test_topk_matches_torch_topk_without_ties():
    s = synthetic.block_scores(2, 3, 16, 16, seed=1)
    got = oracle.mask_from_topk(s, 5, False, False)
    want = torch.zeros_like(s, dtype=torch.uint8).scatter_(-1, torch.topk(s, 5, -1).indices, 1)
    assert np.array_equal(got, want.numpy())
    got = oracle.mask_from_topk(s, 5, True, True)
    want[:, :, -2:, :] = 1
    assert np.array_equal(got, want.tril().numpy())


def test_threshold_and_tril_match_numpy():
    s = synthetic.block_scores(1, 2, 9, 9, seed=2)
    got = oracle.mask_from_threshold(s, 0.6, False, True)
    assert np.array_equal(got, np.tril((s.numpy() > np.float32(0.6)).astype(np.uint8)))


def test_mask_builders_reject_nan():
    s = np.zeros((1, 1, 2, 2), np.float32)
    s[0, 0, 1, 1] = np.nan
    with pytest.raises(ValueError):
        oracle.mask_from_topk(s, 1)
    with pytest.raises(ValueError):
        oracle.mask_from_threshold(s, 0.5)


def test_seed0_active_pair_counts():
    # block selection at seed 0 for the four prefill workloads (tril where the rule asks)
    for name, want in (("C1", 27), ("C2", 9850), ("C3", 120402), ("C4", 262357)):
        cfg = synthetic.PREFILL_CONFIGS[name]
        s = synthetic.block_scores(cfg.B, cfg.H, cfg.nblk, cfg.nblk)
        if cfg.rule == "topk":
            m = oracle.mask_from_topk(s, int(cfg.param), cfg.dense_last, cfg.tril)
        else:
            m = oracle.mask_from_threshold(s, cfg.param, cfg.dense_last, cfg.tril)
        assert int(m.sum()) == want


# ----------------------------------------------------------------- split heuristic

def test_num_splits_hand_worked_cases():
    spec = json.load(open(os.path.join(GOLDEN, "num_splits_cases.json")))
    for c in spec["cases"]:
        assert oracle.num_splits_heuristic(*c["args"]) == c["expect"], c["why"]


def test_decode_num_splits_for_the_decode_shape():
    assert oracle.decode_num_splits(8, 8, 64, 128, 128, 152) == 7
    assert oracle.decode_num_splits(8, 8, 64, 128, 128, 148) == 2


# ----------------------------------------------------------------- XAttention selection

def test_cumulative_pick_worked_example():
    spec = json.load(open(os.path.join(GOLDEN, "find_blocks_chunked_example.json")))
    vals = dict(enumerate(spec["row"]))
    assert oracle.cumulative_pick(vals, spec["threshold"] * sum(spec["row"])) == \
        spec["picked_in_order"]


def test_find_blocks_chunked_keeps_sink_and_diagonal():
    x = np.zeros((1, 1, 3, 3))
    x[0, 0, 2] = [0.1, 0.6, 0.3]
    x[0, 0, 1] = [0.5, 0.5, 0.0]
    x[0, 0, 0] = [1.0, 0.0, 0.0]
    m = oracle.find_blocks_chunked(x, 0.5, causal=True)
    # row 2: sink 0 and diagonal 2 kept; remaining {1: 0.6}: 0 < 0.5 -> take 1
    assert m[0, 0, 2].tolist() == [1, 1, 1]
    # row 1: sink 0, diagonal 1; remaining {2: 0.0}: 0 < 0.5 -> taken (sum still below)
    assert m[0, 0, 1].tolist() == [1, 1, 1]
    # row 0: sink == diagonal; remaining {1: 0, 2: 0}: both taken while the sum stays 0 < 0.5
    assert m[0, 0, 0].tolist() == [1, 1, 1]
    m = oracle.find_blocks_chunked(x, 0.05, causal=False)
    # row 2, non-causal: sink; remaining sorted 1 (0.6), 2 (0.3): take 1, then 0.6 >= 0.03
    assert m[0, 0, 2].tolist() == [1, 1, 0]


# ----------------------------------------------------------------- 128-token mask blocks

@pytest.mark.parametrize("Sq,Sk", [(128, 128), (200, 200), (130, 300), (300, 129)])
@pytest.mark.parametrize("causal", [False, True])
def test_prefill_block128_brute_force(Sq, Sk, causal):
    """A 128-token block mask against SDPA with the token mask built by kron(mask, ones(128))."""
    g = torch.Generator().manual_seed(Sq * 7 + Sk)
    q = torch.randn(1, 2, Sq, 16, generator=g, dtype=torch.float64)
    k = torch.randn(1, 2, Sk, 16, generator=g, dtype=torch.float64)
    v = torch.randn(1, 2, Sk, 16, generator=g, dtype=torch.float64)
    bm = (torch.rand(1, 2, math.ceil(Sq / 128), math.ceil(Sk / 128), generator=g) < 0.6).to(torch.uint8)
    tm = _token_mask(bm, Sq, Sk, causal, block=128)
    got = oracle.prefill(q, k, v, bm, causal, block=128)
    empty = ~tm.any(-1).numpy()
    assert np.all(got[empty] == 0.0)
    if (~empty).any():
        want = _sdpa(q, k, v, tm).numpy()
        assert np.abs(got[~empty] - want[~empty]).max() <= 1e-12


def test_prefill_block128_equals_its_64_expansion():
    """Each 128-token entry is the four 64-token entries it covers: same token sets, so the
    oracle gives bit-identical results for the two forms."""
    g = torch.Generator().manual_seed(5)
    Sq, Sk = 333, 450
    q, k, v = synthetic.qkv(1, 3, Sq, Sk, 64, torch.bfloat16, seed=5)
    bm = (torch.rand(1, 3, math.ceil(Sq / 128), math.ceil(Sk / 128), generator=g) < 0.5).to(torch.uint8)
    m64 = bm.repeat_interleave(2, dim=2).repeat_interleave(2, dim=3)[:, :, :math.ceil(Sq / 64), :math.ceil(Sk / 64)]
    for causal in (False, True):
        a = oracle.prefill(q, k, v, bm, causal, block=128)
        b = oracle.prefill(q, k, v, m64, causal, block=64)
        assert np.array_equal(a, b)

"""GPU parity of bsattn_prefill (through the C ABI) against the fp64 oracle.

Tolerance (fixed by the task for this method): max |err| <= 1e-2 for fp16 inputs and
<= 2e-2 for bf16 inputs, both sides fed the same rounded inputs and the same block mask
(built by the oracle's builder).  Every case, the full-size workloads included, compares
every output element.
"""
import math

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


def _run(bsa, q, k, v, mask, causal):
    dev = torch.device("cuda")
    out = bsa.bsattn_prefill(q.to(dev), k.to(dev), v.to(dev), torch.as_tensor(mask).to(dev),
                             causal)
    torch.cuda.synchronize()
    return out.cpu()


def _err(got, want):
    return float(np.abs(got.double().numpy() - want).max()) if want.size else 0.0


CASES = [
    # B, H, Sq, Sk, d, dtype, causal, density
    (1, 1, 64, 64, 64, torch.float16, True, 1.0),
    (1, 1, 64, 64, 128, torch.bfloat16, False, 1.0),
    (1, 2, 130, 130, 64, torch.float16, True, 0.6),
    (2, 3, 200, 200, 128, torch.bfloat16, True, 0.5),
    (1, 2, 256, 256, 128, torch.bfloat16, False, 0.5),
    (1, 1, 1, 1, 64, torch.float16, False, 1.0),
    (1, 1, 63, 63, 128, torch.bfloat16, True, 1.0),
    (1, 1, 65, 65, 64, torch.float16, False, 0.7),
    (2, 2, 512, 512, 64, torch.float16, True, 0.3),
    (1, 2, 700, 700, 128, torch.bfloat16, True, 0.4),
    (1, 2, 700, 700, 64, torch.bfloat16, False, 0.25),
    (1, 1, 1000, 1000, 128, torch.float16, True, 1.0),
    # Sq != Sk: bottom-right causal alignment, and plain non-causal
    (1, 2, 100, 300, 64, torch.float16, True, 0.8),
    (1, 2, 300, 100, 128, torch.bfloat16, True, 0.8),
    (1, 1, 64, 1000, 128, torch.bfloat16, False, 0.5),
]


@pytest.mark.parametrize("B,H,Sq,Sk,d,dtype,causal,density", CASES)
def test_prefill_small_cases(bsa, B, H, Sq, Sk, d, dtype, causal, density):
    q, k, v = synthetic.qkv(B, H, Sq, Sk, d, dtype, seed=Sq + d)
    mask = synthetic.random_block_mask(B, H, math.ceil(Sq / 64), math.ceil(Sk / 64), density,
                                       seed=Sk)
    got = _run(bsa, q, k, v, mask, causal)
    want = oracle.prefill(q, k, v, mask, causal)
    assert _err(got, want) <= TOL[dtype]
    # rows the oracle says are exactly zero are exactly zero on the GPU too
    zero_rows = np.all(want == 0.0, axis=-1)
    assert np.all(got.double().numpy()[zero_rows] == 0.0)


def test_prefill_all_masked_is_zero(bsa):
    q, k, v = synthetic.qkv(1, 2, 300, 300, 128, torch.bfloat16, seed=1)
    mask = torch.zeros(1, 2, 5, 5, dtype=torch.uint8)
    got = _run(bsa, q, k, v, mask, True)
    assert torch.count_nonzero(got) == 0


def test_prefill_above_diagonal_entries_ignored_when_causal(bsa):
    q, k, v = synthetic.qkv(1, 2, 256, 256, 64, torch.float16, seed=2)
    mask = synthetic.random_block_mask(1, 2, 4, 4, 0.5, seed=2)
    upper = mask | torch.ones(4, 4, dtype=torch.uint8).triu(1)
    assert torch.equal(_run(bsa, q, k, v, mask, True), _run(bsa, q, k, v, upper, True))


def test_prefill_is_deterministic(bsa):
    q, k, v = synthetic.qkv(1, 4, 1024, 1024, 128, torch.bfloat16, seed=3)
    mask = synthetic.random_block_mask(1, 4, 16, 16, 0.5, seed=3)
    a = _run(bsa, q, k, v, mask, True)
    b = _run(bsa, q, k, v, mask, True)
    assert torch.equal(a, b)


def test_c1_full_oracle(bsa):
    cfg = synthetic.PREFILL_CONFIGS["C1"]
    q, k, v, scores = synthetic.prefill_inputs(cfg)
    mask = oracle.mask_from_topk(scores, int(cfg.param), cfg.dense_last, cfg.tril)
    got = _run(bsa, q, k, v, mask, cfg.causal)
    want = oracle.prefill(q, k, v, mask, cfg.causal)
    assert _err(got, want) <= TOL[cfg.dtype]


def _workload_mask(cfg, scores):
    if cfg.rule == "topk":
        return oracle.mask_from_topk(scores, int(cfg.param), cfg.dense_last, cfg.tril)
    return oracle.mask_from_threshold(scores, cfg.param, cfg.dense_last, cfg.tril)


@pytest.mark.parametrize("name", ["C2", "C3", "C4"])
def test_full_size_workloads_every_element(bsa, name):
    """The benchmark's workloads at full size, in the benchmark's launch configuration,
    compared with the fp64 oracle on every output element (C3: 67 M, C4: 33.5 M values)."""
    cfg = synthetic.PREFILL_CONFIGS[name]
    q, k, v, scores = synthetic.prefill_inputs(cfg)
    mask = _workload_mask(cfg, scores)
    got = _run(bsa, q, k, v, mask, cfg.causal)
    want = oracle.prefill(q, k, v, mask, cfg.causal)
    assert torch.isfinite(got.float()).all()
    assert _err(got, want) <= TOL[cfg.dtype]
    zero_rows = np.all(want == 0.0, axis=-1)
    assert np.all(got.double().numpy()[zero_rows] == 0.0)


def _used_columns_mask(B, H, nq, nk, density, seed, causal):
    """A block mask whose rows only ever select a random half of the key blocks of each
    head ("used" columns), plus, when causal, every entry above the diagonal set (those are
    ignored by the causal rule).  Returns (mask, used [B, H, nk] bool)."""
    g = torch.Generator().manual_seed(seed)
    used = torch.rand(B, H, nk, generator=g) < 0.5
    used[..., 0] = True
    mask = (torch.rand(B, H, nq, nk, generator=g) < density) & used[:, :, None, :]
    if causal:
        above = torch.ones(nq, nk, dtype=torch.bool).triu(1 + max(0, nk - nq))
        mask |= above
    return mask.to(torch.uint8), used


def _poison_unused(k, v, used):
    """NaN in every K and V row of a key block no visited entry selects."""
    kp, vp = k.clone(), v.clone()
    B, H, Sk, _ = k.shape
    for b in range(B):
        for h in range(H):
            for kb in torch.nonzero(~used[b, h]).flatten().tolist():
                kp[b, h, kb * 64:(kb + 1) * 64] = float("nan")
                vp[b, h, kb * 64:(kb + 1) * 64] = float("nan")
    return kp, vp


@pytest.mark.parametrize("d,dtype,causal", [(128, torch.bfloat16, True), (64, torch.float16, True),
                                            (128, torch.float16, False), (64, torch.bfloat16, False)])
def test_unselected_tiles_are_never_loaded(bsa, d, dtype, causal):
    """Masked blocks are skipped without being loaded (the guide's section 4.4: the skipping
    is the whole benefit).  Every K/V tile that no visited mask entry selects -- including
    tiles referenced only by entries above the causal diagonal -- holds NaN; the output is
    bit-identical to the run on clean K/V and matches the oracle."""
    B, H, S = 2, 3, 1500                       # 24 key blocks, ragged tail of 28 keys
    q, k, v = synthetic.qkv(B, H, S, S, d, dtype, seed=31 + d)
    nb = math.ceil(S / 64)
    mask, used = _used_columns_mask(B, H, nb, nb, 0.5, seed=d, causal=causal)
    kp, vp = _poison_unused(k, v, used)
    clean = _run(bsa, q, k, v, mask, causal)
    poisoned = _run(bsa, q, kp, vp, mask, causal)
    assert torch.equal(clean, poisoned)
    want = oracle.prefill(q, k, v, mask, causal)
    assert _err(poisoned, want) <= TOL[dtype]


@pytest.mark.parametrize("name", ["C3", "C4"])
def test_unselected_tiles_are_never_loaded_full_size(bsa, name):
    """The same at a full workload's shape and launch configuration: its mask restricted to a
    random half of each head's key blocks; every other K/V tile is NaN; output bit-identical to
    the clean run."""
    cfg = synthetic.PREFILL_CONFIGS[name]
    q, k, v, scores = synthetic.prefill_inputs(cfg)
    mask = torch.as_tensor(_workload_mask(cfg, scores))
    g = torch.Generator().manual_seed(9)
    used = torch.rand(cfg.B, cfg.H, cfg.nblk, generator=g) < 0.5
    mask = (mask.bool() & used[:, :, None, :]).to(torch.uint8)
    kp, vp = _poison_unused(k, v, used)
    clean = _run(bsa, q, k, v, mask, cfg.causal)
    poisoned = _run(bsa, q, kp, vp, mask, cfg.causal)
    assert torch.isfinite(clean.float()).all()
    assert torch.equal(clean, poisoned)


@pytest.mark.parametrize("d,dtype,causal", [(64, torch.float16, True), (64, torch.bfloat16, False),
                                            (128, torch.bfloat16, True), (128, torch.float16, False)])
def test_prefill_rescale_path(bsa, d, dtype, causal):
    """Scores that grow by far more than 2^8 (in exp2 units) from one key block to the next:
    the online softmax must rescale the accumulated output (the kernels do so lazily, only
    past that growth), and the result still matches the oracle."""
    B, H, S = 1, 3, 900
    q, k, v = synthetic.qkv(B, H, S, S, d, dtype, seed=41 + d)
    nb = math.ceil(S / 64)
    scale = torch.tensor([4.0 * kb + 1.0 for kb in range(nb)]).repeat_interleave(64)[:S]
    k = (k.float() * scale[None, None, :, None]).to(dtype)
    mask = synthetic.random_block_mask(B, H, nb, nb, 0.6, seed=d)
    got = _run(bsa, q, k, v, mask, causal)
    want = oracle.prefill(q, k, v, mask, causal)
    assert _err(got, want) <= TOL[dtype]


@pytest.mark.parametrize("d", [128, 64])
def test_timeout_path_reports_and_recovers(bsa, d):
    """A wait budget of 0 makes the kernels' bounded waits expire: the call must record
    BSATTN_ERR_TIMEOUT in the status word and leave the context usable."""
    q, k, v = synthetic.qkv(2, 8, 2048, 2048, d, torch.bfloat16, seed=4)
    mask = synthetic.random_block_mask(2, 8, 32, 32, 0.5, seed=4)
    dev = torch.device("cuda")
    qd, kd, vd, md = q.to(dev), k.to(dev), v.to(dev), mask.to(dev)
    ws = bsa.workspace(dev, "prefill", 256)
    bsa.bsattn_get_device_status(ws)            # clear
    try:
        bsa.bsattn_set_wait_budget_ns(0)
        bsa.bsattn_prefill(qd, kd, vd, md, True)
        torch.cuda.synchronize()
    finally:
        bsa.bsattn_set_wait_budget_ns(2_000_000_000)
    status = bsa.bsattn_get_device_status(ws)
    assert status & bsa.BSATTN_ERR_TIMEOUT
    got = bsa.bsattn_prefill(qd, kd, vd, md, True).cpu()
    assert bsa.bsattn_get_device_status(ws) == 0
    want = oracle.prefill(q[:1, :2], k[:1, :2], v[:1, :2], mask[:1, :2], True)
    assert _err(got[:1, :2], want) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("d,dtype", [(128, torch.bfloat16), (64, torch.float16)])
def test_long_rows_split_across_ctas(bsa, d, dtype):
    """Rows visiting more than 96 key blocks are split into parts run by different CTAs and
    merged by log-sum-exp once rows can span 1024+ key blocks (64K+ keys); the result matches
    the oracle, matches an unsplit run (minimal workspace) within rounding, and is the same
    from run to run."""
    dev = torch.device("cuda")
    B, H, S = 1, 2, 66000
    q, k, v = synthetic.qkv(B, H, S, S, d, dtype, seed=21)
    nb = math.ceil(S / 64)
    # 5% of the blocks, plus the last two query-block rows dense (1031 and 1032 blocks): only
    # those rows are split (17 parts each), well within the 2048 partial slots
    mask = synthetic.random_block_mask(B, H, nb, nb, 0.05, seed=21)
    mask[:, :, -2:, :] = 1
    args = [t.to(dev) for t in (q, k, v, mask)]
    split = bsa.bsattn_prefill(*args, True).cpu()
    again = bsa.bsattn_prefill(*args, True).cpu()
    assert torch.equal(split, again)
    small_ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    whole = bsa.bsattn_prefill(*args, True, ws=small_ws).cpu()
    assert float((split.float() - whole.float()).abs().max()) <= TOL[dtype]
    # whole query blocks: the first, one in the middle, and the two dense last ones (split)
    rows = list(range(0, 64)) + list(range(40000, 40064)) + list(range(65920, S))
    for h in range(H):
        want = oracle.prefill_rows(q, k, v, mask, True, 0, h, rows)
        assert _err(split[0, h, rows], want) <= TOL[dtype]
        assert _err(whole[0, h, rows], want) <= TOL[dtype]


@pytest.mark.parametrize("S,d", [(96000, 128), (258000, 64)])
def test_wide_masks(bsa, S, d):
    """The widest masks: at d = 128 more than 1304 key blocks, too wide for the deeper rings'
    shared memory, run the kernel with two-stage K/V rings; at d = 64 the deeper rings take every
    width the library accepts (here 4032 key blocks, rows split across CTAs).  Sampled rows match
    the oracle."""
    dev = torch.device("cuda")
    dtype = torch.bfloat16 if d == 128 else torch.float16
    q, k, v = synthetic.qkv(1, 1, S, S, d, dtype, seed=23)
    nb = math.ceil(S / 64)
    mask = synthetic.random_block_mask(1, 1, nb, nb, 0.02, seed=23)
    got = bsa.bsattn_prefill(*[t.to(dev) for t in (q, k, v, mask)], True).cpu()
    rows = list(range(0, 64)) + list(range(S // 2 - 32, S // 2 + 32)) + list(range(S - 64, S))
    want = oracle.prefill_rows(q, k, v, mask, True, 0, 0, rows)
    assert _err(got[0, 0, rows], want) <= TOL[dtype]


BS128_CASES = [
    # B, H, Sq, Sk, d, dtype, causal, density (of the 128-token block mask)
    (1, 2, 128, 128, 64, torch.float16, True, 0.6),
    (2, 2, 300, 300, 128, torch.bfloat16, True, 0.5),
    (1, 2, 130, 400, 128, torch.bfloat16, True, 0.7),      # Sq < Sk, bottom-right causal
    (1, 2, 400, 130, 64, torch.float16, True, 0.7),        # Sq > Sk: early rows see no key
    (1, 3, 700, 700, 64, torch.float16, False, 0.4),
    (1, 1, 1000, 1000, 128, torch.bfloat16, True, 1.0),
    (2, 3, 1111, 1111, 128, torch.float16, False, 0.3),
    (1, 1, 1, 1, 64, torch.bfloat16, True, 1.0),
    (1, 2, 127, 129, 64, torch.bfloat16, False, 1.0),
    # more than 256 key tiles at d = 128: the one-CTA-per-SM layout
    (1, 2, 20000, 20000, 128, torch.bfloat16, True, 0.08),
]


@pytest.mark.parametrize("B,H,Sq,Sk,d,dtype,causal,density", BS128_CASES)
def test_prefill_block128(bsa, B, H, Sq, Sk, d, dtype, causal, density):
    """128-token mask blocks (the 128-row kernel, full-rate M = 128 tiles): parity with the
    oracle at block 128, and agreement with the same mask expanded to 64-token blocks (the 64-row
    kernel) within the tolerance; rows the oracle says are zero are exactly zero."""
    q, k, v = synthetic.qkv(B, H, Sq, Sk, d, dtype, seed=Sq + 3 * d)
    mask = synthetic.random_block_mask(B, H, math.ceil(Sq / 128), math.ceil(Sk / 128), density,
                                       seed=Sk + 1)
    dev = torch.device("cuda")
    got = bsa.bsattn_prefill(q.to(dev), k.to(dev), v.to(dev), mask.to(dev), causal,
                             block_size=128).cpu()
    want = oracle.prefill(q, k, v, mask, causal, block=128)
    assert _err(got, want) <= TOL[dtype]
    zero_rows = np.all(want == 0.0, axis=-1)
    assert np.all(got.double().numpy()[zero_rows] == 0.0)
    m64 = mask.repeat_interleave(2, dim=2).repeat_interleave(2, dim=3)
    m64 = m64[:, :, :math.ceil(Sq / 64), :math.ceil(Sk / 64)].contiguous()
    assert float((got.float() - _run(bsa, q, k, v, m64, causal).float()).abs().max()) <= TOL[dtype]


def _block128_workload(name):
    """A full workload's shape and mask rule on 128-token blocks (scores [B, H, S/128, S/128])."""
    cfg = synthetic.PREFILL_CONFIGS[name]
    q, k, v, _ = synthetic.prefill_inputs(cfg)
    n = math.ceil(cfg.S / 128)
    scores = synthetic.block_scores(cfg.B, cfg.H, n, n, seed=0)
    return cfg, q, k, v, torch.as_tensor(_workload_mask(cfg, scores))


@pytest.mark.parametrize("name", ["C3", "C4"])
def test_block128_full_size_every_element(bsa, name):
    """C3 and C4 shapes with their mask rules on 128-token blocks, through the 128-row kernel,
    against the oracle on every output element."""
    cfg, q, k, v, mask = _block128_workload(name)
    dev = torch.device("cuda")
    got = bsa.bsattn_prefill(q.to(dev), k.to(dev), v.to(dev), mask.to(dev), cfg.causal,
                             block_size=128).cpu()
    want = oracle.prefill(q, k, v, mask, cfg.causal, block=128)
    assert torch.isfinite(got.float()).all()
    assert _err(got, want) <= TOL[cfg.dtype]


@pytest.mark.parametrize("d,dtype,causal", [(128, torch.bfloat16, True), (64, torch.float16, False)])
def test_block128_unselected_tiles_are_never_loaded(bsa, d, dtype, causal):
    """The 128-row kernel skips unselected blocks without loading them: NaN in every K/V block
    no visited 128-token entry selects leaves the output bit-identical to the clean run."""
    B, H, S = 1, 3, 1700
    q, k, v = synthetic.qkv(B, H, S, S, d, dtype, seed=51 + d)
    nb = math.ceil(S / 128)
    mask, used = _used_columns_mask(B, H, nb, nb, 0.5, seed=d + 1, causal=causal)
    used64 = used.repeat_interleave(2, dim=2)[:, :, :math.ceil(S / 64)]
    kp, vp = _poison_unused(k, v, used64)
    dev = torch.device("cuda")
    run = lambda kk, vv: bsa.bsattn_prefill(q.to(dev), kk.to(dev), vv.to(dev), mask.to(dev), causal,
                                            block_size=128).cpu()
    clean, poisoned = run(k, v), run(kp, vp)
    assert torch.equal(clean, poisoned)
    assert _err(poisoned, oracle.prefill(q, k, v, mask, causal, block=128)) <= TOL[dtype]


@pytest.mark.parametrize("d", [128, 64])
def test_block128_timeout_path_reports_and_recovers(bsa, d):
    """The 128-row kernel's bounded waits expire with a budget of 0: BSATTN_ERR_TIMEOUT is
    recorded and the next call is correct."""
    q, k, v = synthetic.qkv(2, 8, 2048, 2048, d, torch.bfloat16, seed=6)
    mask = synthetic.random_block_mask(2, 8, 16, 16, 0.5, seed=6)
    dev = torch.device("cuda")
    qd, kd, vd, md = q.to(dev), k.to(dev), v.to(dev), mask.to(dev)
    ws = bsa.workspace(dev, "prefill", 256)
    bsa.bsattn_get_device_status(ws)
    try:
        bsa.bsattn_set_wait_budget_ns(0)
        bsa.bsattn_prefill(qd, kd, vd, md, True, block_size=128)
        torch.cuda.synchronize()
    finally:
        bsa.bsattn_set_wait_budget_ns(2_000_000_000)
    assert bsa.bsattn_get_device_status(ws) & bsa.BSATTN_ERR_TIMEOUT
    got = bsa.bsattn_prefill(qd, kd, vd, md, True, block_size=128).cpu()
    assert bsa.bsattn_get_device_status(ws) == 0
    want = oracle.prefill(q[:1, :2], k[:1, :2], v[:1, :2], mask[:1, :2], True, block=128)
    assert _err(got[:1, :2], want) <= TOL[torch.bfloat16]

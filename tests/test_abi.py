"""C-ABI library checks that need no GPU: it loads, exports every function the public header
declares, its host-side mask builders and split-count rule agree bit-for-bit with the
oracle's independent versions, and argument checks fail before anything is launched."""
import ctypes
import json
import os
import re

import numpy as np
import pytest
import torch

import oracle
import synthetic
import block_sparse_attention_gb300 as bsa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b(bsattn_[a-z0-9_]+)\s*\(", text))
    return names


def test_library_exports_every_declared_symbol():
    lib = bsa.load()
    declared = _declared_functions()
    assert len(declared) >= 12
    missing = [n for n in sorted(declared) if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings():
    assert bsa.bsattn_status_string(0) == "BSATTN_OK"
    assert bsa.bsattn_status_string(bsa.BSATTN_ERR_TIMEOUT | bsa.BSATTN_ERR_BAD_INDEX) == \
        "BSATTN_ERR_TIMEOUT|BSATTN_ERR_BAD_INDEX"
    assert "sm_103a" in bsa.bsattn_version()


# ----------------------------------------------------------------- mask builders vs oracle

@pytest.mark.parametrize("dense_last", [False, True])
@pytest.mark.parametrize("tril", [False, True])
def test_topk_builder_bit_exact(dense_last, tril):
    s = synthetic.block_scores(2, 3, 17, 17, seed=4)
    for k in (0, 1, 3, 16, 17, 40):
        got = bsa.bsattn_mask_from_topk(s, k, dense_last, tril).numpy()
        assert np.array_equal(got, oracle.mask_from_topk(s, k, dense_last, tril)), k


def test_topk_builder_ties_and_rectangles():
    g = torch.Generator().manual_seed(3)
    s = torch.randint(0, 4, (2, 2, 9, 13), generator=g).float() / 4     # many ties
    s[0, 0, 0, :] = 0.0
    s[0, 0, 1, 3] = -0.0
    for k in (1, 2, 5, 13):
        for dl in (False, True):
            got = bsa.bsattn_mask_from_topk(s, k, dl, True).numpy()
            assert np.array_equal(got, oracle.mask_from_topk(s, k, dl, True))


def test_threshold_builder_bit_exact():
    s = synthetic.block_scores(1, 4, 33, 33, seed=8)
    s[0, 0, 0, :4] = 0.75                       # equality: must be dropped
    for thr in (0.0, 0.5, 0.75, 0.9, 1.0):
        for dl in (False, True):
            for tril in (False, True):
                got = bsa.bsattn_mask_from_threshold(s, thr, dl, tril).numpy()
                assert np.array_equal(got, oracle.mask_from_threshold(s, thr, dl, tril))


def test_builders_on_the_workload_masks():
    for name, cfg in synthetic.PREFILL_CONFIGS.items():
        s = synthetic.block_scores(cfg.B, cfg.H, cfg.nblk, cfg.nblk)
        if cfg.rule == "topk":
            got = bsa.bsattn_mask_from_topk(s, int(cfg.param), cfg.dense_last, cfg.tril)
            want = oracle.mask_from_topk(s, int(cfg.param), cfg.dense_last, cfg.tril)
        else:
            got = bsa.bsattn_mask_from_threshold(s, cfg.param, cfg.dense_last, cfg.tril)
            want = oracle.mask_from_threshold(s, cfg.param, cfg.dense_last, cfg.tril)
        assert np.array_equal(got.numpy(), want), name


def test_builders_golden_and_nan():
    spec = json.load(open(os.path.join(GOLDEN, "mask_builders_4x4.json")))
    s = torch.tensor(spec["scores"], dtype=torch.float32)
    for c in spec["cases"]:
        fn = bsa.bsattn_mask_from_topk if c["rule"] == "topk" else bsa.bsattn_mask_from_threshold
        got = fn(s, c["param"], c["dense_last"], c["tril"])[0, 0].numpy()
        assert np.array_equal(got, np.array(c["expect"], np.uint8)), c["why"]
    s[0, 0, 2, 2] = float("nan")
    with pytest.raises(bsa.BsattnError):
        bsa.bsattn_mask_from_topk(s, 2)
    with pytest.raises(bsa.BsattnError):
        bsa.bsattn_mask_from_threshold(s, 0.5)


# ----------------------------------------------------------------- split rule vs oracle

def test_num_splits_heuristic_golden():
    spec = json.load(open(os.path.join(GOLDEN, "num_splits_cases.json")))
    for c in spec["cases"]:
        assert bsa.bsattn_num_splits_heuristic(*c["args"]) == c["expect"], c["why"]


def test_num_splits_heuristic_matches_oracle_random():
    rng = np.random.default_rng(0)
    for _ in range(3000):
        args = (int(rng.integers(1, 400)), int(rng.integers(1, 200)), int(rng.integers(1, 300)),
                int(rng.integers(1, 800)), int(rng.integers(1, 2**31)) * int(rng.integers(1, 4)),
                bool(rng.integers(0, 2)), int(rng.integers(1, 160)))
        assert bsa.bsattn_num_splits_heuristic(*args) == oracle.num_splits_heuristic(*args), args


def test_default_splits_shape():
    # without a GPU the library assumes 4 resident decode CTAs per SM: at most one wave
    # (64 groups x s <= 608), then the fewest splits with the same longest slice
    s = bsa.bsattn_decode_default_splits(8, 8, 64, 128, 152)
    assert s == 8 and 64 * s <= 4 * 152
    assert bsa.bsattn_decode_default_splits(1, 1, 3, 128, 152) == 3
    for groups, max_sel in ((64, 64), (64, 50), (16, 64), (300, 64), (7, 1000)):
        s = bsa.bsattn_decode_default_splits(groups, 1, max_sel, 128, 152)
        cap = max(1, min(64, max_sel, 4 * 152 // groups))
        assert 1 <= s <= cap
        assert -(-max_sel // s) == -(-max_sel // cap)          # longest slice as short as possible
        assert s == 1 or -(-max_sel // (s - 1)) > -(-max_sel // s)   # and the fewest splits for it


# ----------------------------------------------------------------- argument checks (no launch)

def _call_prefill(lib, **kw):
    a = dict(q=1 << 12, k=1 << 12, v=1 << 12, mask=1 << 12, causal=1, out=1 << 12, B=1, H=1, Sq=64,
             Sk=64, d=64, dtype=0, ws=1 << 12, ws_bytes=256, stream=None)
    a.update(kw)
    return lib.bsattn_prefill(a["q"], a["k"], a["v"], a["mask"], a["causal"], a["out"], a["B"],
                              a["H"], a["Sq"], a["Sk"], a["d"], a["dtype"], a["ws"], a["ws_bytes"],
                              a["stream"])


def test_prefill_rejects_bad_arguments_without_launching():
    lib = bsa.load()
    assert _call_prefill(lib, d=96) == bsa.BSATTN_ERR_UNSUPPORTED
    assert _call_prefill(lib, dtype=5) == bsa.BSATTN_ERR_UNSUPPORTED
    assert _call_prefill(lib, ws=None) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_prefill(lib, ws_bytes=8) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_prefill(lib, q=None) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_prefill(lib, q=(1 << 12) + 2) == bsa.BSATTN_ERR_INVALID_ARG   # misaligned
    assert _call_prefill(lib, B=-1) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_prefill(lib, Sq=0) == bsa.BSATTN_OK                          # nothing to do
    for bs, want in ((32, bsa.BSATTN_ERR_UNSUPPORTED), (96, bsa.BSATTN_ERR_UNSUPPORTED)):
        assert lib.bsattn_prefill_bs(1 << 12, 1 << 12, 1 << 12, 1 << 12, bs, 1, 1 << 12, 1, 1, 64,
                                     64, 64, 0, 1 << 12, 256, None) == want


def _call_decode(lib, **kw):
    a = dict(q=1 << 12, k=1 << 12, v=1 << 12, sl=1 << 12, idx=1 << 12, ns=0, out=1 << 12, B=1, Hq=4,
             Hkv=1, Smax=64, d=128, max_sel=1, dtype=1, ws=1 << 12, ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return lib.bsattn_decode_varlen(a["q"], a["k"], a["v"], a["sl"], a["idx"], a["ns"], a["out"],
                                    a["B"], a["Hq"], a["Hkv"], a["Smax"], a["d"], a["max_sel"],
                                    a["dtype"], a["ws"], a["ws_bytes"], a["stream"])


def test_decode_rejects_bad_arguments_without_launching():
    lib = bsa.load()
    assert _call_decode(lib, Hq=6, Hkv=4) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_decode(lib, Hq=32, Hkv=2) == bsa.BSATTN_ERR_UNSUPPORTED     # group of 16
    assert _call_decode(lib, d=80) == bsa.BSATTN_ERR_UNSUPPORTED
    assert _call_decode(lib, ns=-1) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_decode(lib, ws=None) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_decode(lib, ws_bytes=16) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_decode(lib, k=None) == bsa.BSATTN_ERR_INVALID_ARG
    assert _call_decode(lib, B=0) == bsa.BSATTN_OK


def test_noalloc_decode_rejects_shapes_beyond_its_scratch_without_launching():
    """The allocation-free decode keeps its split partials in a fixed 8 MiB array: a shape
    whose decode workspace exceeds it is refused before any device work."""
    lib = bsa.load()
    f = lib.bsattn_decode_varlen_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, P]
    f.restype = I
    B, Hq, Hkv, d, max_sel, ns = 64, 64, 8, 128, 64, 64
    assert bsa.bsattn_decode_workspace_size(B, Hq, Hkv, d, max_sel, ns) > (8 << 20)
    x = 1 << 12
    assert f(x, x, x, x, x, ns, x, B, Hq, Hkv, 65536, d, max_sel, 1, None) == \
        bsa.BSATTN_ERR_UNSUPPORTED
    assert f(x, x, x, x, x, -1, x, 1, 4, 1, 64, d, 1, 1, None) == bsa.BSATTN_ERR_INVALID_ARG


def test_workspace_sizes_grow_with_splits():
    a = bsa.bsattn_decode_workspace_size(8, 32, 8, 128, 64, 2)
    b = bsa.bsattn_decode_workspace_size(8, 32, 8, 128, 64, 16)
    assert b > a >= 8 * 32 * 2 * 128 * 4
    assert bsa.bsattn_prefill_workspace_size(2, 8, 4096, 4096) >= 4


# ----------------------------------------------------------------- XAttention selection rule

def test_cumulative_threshold_builder_worked_example():
    spec = json.load(open(os.path.join(GOLDEN, "find_blocks_chunked_example.json")))
    row = torch.tensor(spec["row"], dtype=torch.float32).view(1, 1, 1, -1)
    got = bsa.bsattn_mask_from_cumulative_threshold(row, spec["threshold"], causal=False)
    # the sink block is kept as well as the four picks 2, 1, 3, 4 of the example
    assert got[0, 0, 0].tolist() == [1, 1, 1, 1, 1]
    assert np.array_equal(got.numpy(), oracle.find_blocks_chunked(row.numpy(), spec["threshold"], False))


@pytest.mark.parametrize("causal", [False, True])
def test_cumulative_threshold_builder_matches_oracle(causal):
    g = torch.Generator().manual_seed(11)
    x = torch.rand(2, 3, 12, 12, generator=g) ** 3          # skewed weights, like softmax sums
    x[0, 0, 5] = 0.25                                        # ties
    for thr in (0.3, 0.5, 0.9, 0.95, 1.0):
        got = bsa.bsattn_mask_from_cumulative_threshold(x, thr, causal)
        assert np.array_equal(got.numpy(), oracle.find_blocks_chunked(x.numpy(), thr, causal)), thr
    x[1, 2, 3, 4] = float("nan")
    with pytest.raises(bsa.BsattnError):
        bsa.bsattn_mask_from_cumulative_threshold(x, 0.9, causal)

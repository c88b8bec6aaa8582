"""The allocation-free decode entry point (bsattn_decode_varlen_noalloc), called through the
C ABI, must give the same output as bsattn_decode_varlen on the same inputs, and match the
fp64 oracle, on two calls in a row (its scratch array keeps the previous call's contents, so
the second call checks that it starts clean).  It exists for callers that cannot allocate
device memory when they attend, e.g. code running inside a custom allocator or memory pool,
which must not re-enter the allocator it implements."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]

TOL = {torch.float16: 1e-2, torch.bfloat16: 2e-2}


@pytest.mark.parametrize("d,dtype,ns", [(128, torch.bfloat16, 4), (128, torch.bfloat16, 0),
                                        (64, torch.float16, 3)])
def test_noalloc_decode_matches_decode_and_oracle_twice(d, dtype, ns):
    import block_sparse_attention_gb300 as bsa
    lib = bsa.load()
    f = lib.bsattn_decode_varlen_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, P]
    f.restype = I

    dev = torch.device("cuda", torch.cuda.current_device())
    B, Hq, Hkv, Smax, nsel = 4, 16, 4, 4096, 16
    sl, idx = synthetic.decode_selection(B, Hkv, 1000, Smax, nsel, nsel, seed=3)
    q, k, v = synthetic.decode_qkv(B, Hq, Hkv, Smax, d, dtype, sl, seed=3)
    oracle_out = oracle.decode_varlen(q, k, v, sl, idx)
    qd, kd, vd, sld, idxd = (t.to(dev) for t in (q, k, v, sl, idx))
    want = bsa.bsattn_decode_varlen(qd, kd, vd, sld, idxd, ns)
    code = 1 if dtype == torch.bfloat16 else 0
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):
        out = torch.full_like(qd, float("nan"))
        rc = f(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), sld.data_ptr(), idxd.data_ptr(), ns,
               out.data_ptr(), B, Hq, Hkv, Smax, d, nsel, code, stream)
        assert rc == 0, bsa.bsattn_status_string(rc)
        torch.cuda.synchronize()
        assert float((out.float() - want.float()).abs().max()) <= TOL[dtype]
        err = float(np.abs(out.cpu().double().numpy() - oracle_out).max())
        assert err <= TOL[dtype], err
    # the same call through the Python binding
    out = bsa.bsattn_decode_varlen_noalloc(qd, kd, vd, sld, idxd, ns)
    assert bsa.bsattn_decode_noalloc_status() == 0
    assert float((out.float() - want.float()).abs().max()) <= TOL[dtype]


def test_noalloc_status_reports_bad_index_and_expired_wait():
    """Device-detected conditions of the allocation-free decode land in its array's status word,
    read and cleared with bsattn_decode_noalloc_status: an index past the sequence end is skipped
    and sets BSATTN_ERR_BAD_INDEX (the output still matches the oracle), a wait budget of 0 sets
    BSATTN_ERR_TIMEOUT, and a clean call reports nothing."""
    import block_sparse_attention_gb300 as bsa
    lib = bsa.load()
    f = lib.bsattn_decode_varlen_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, P]
    f.restype = I
    status = lib.bsattn_decode_noalloc_status
    status.argtypes = [P]
    status.restype = I

    dev = torch.device("cuda", torch.cuda.current_device())
    B, Hq, Hkv, Smax, nsel, d, dtype = 4, 16, 4, 4096, 16, 128, torch.bfloat16
    sl, idx = synthetic.decode_selection(B, Hkv, 1000, Smax, nsel, nsel, seed=5)
    q, k, v = synthetic.decode_qkv(B, Hq, Hkv, Smax, d, dtype, sl, seed=5)
    bad = idx.clone()
    bad[0, 0, 0] = (int(sl[0]) + 63) // 64          # the first block wholly past sequence 0's end
    qd, kd, vd, sld = (t.to(dev) for t in (q, k, v, sl))
    stream = torch.cuda.current_stream(dev).cuda_stream

    def call(index):
        out = torch.full_like(qd, float("nan"))
        rc = f(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), sld.data_ptr(), index.data_ptr(), 4,
               out.data_ptr(), B, Hq, Hkv, Smax, d, nsel, 1, stream)
        assert rc == 0, bsa.bsattn_status_string(rc)
        return out

    idxd, badd = idx.to(dev), bad.to(dev)
    call(idxd)
    assert status(stream) == 0
    got = call(badd)
    assert status(stream) & bsa.BSATTN_ERR_BAD_INDEX
    assert status(stream) == 0                      # the read cleared it
    err = float(np.abs(got.cpu().double().numpy() - oracle.decode_varlen(q, k, v, sl, bad)).max())
    assert err <= TOL[dtype], err
    try:
        bsa.bsattn_set_wait_budget_ns(0)
        call(idxd)
        torch.cuda.synchronize()
    finally:
        bsa.bsattn_set_wait_budget_ns(2_000_000_000)
    assert status(stream) & bsa.BSATTN_ERR_TIMEOUT
    got = call(idxd)
    assert status(stream) == 0
    err = float(np.abs(got.cpu().double().numpy() - oracle.decode_varlen(q, k, v, sl, idx)).max())
    assert err <= TOL[dtype], err

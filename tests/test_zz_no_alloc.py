"""The allocation-free decode entry point (bsattn_decode_varlen_noalloc), called through the
C ABI, must give the same output as bsattn_decode_varlen on the same inputs, on two calls
in a row (its scratch array keeps the previous call's contents, so the second call checks
that it starts clean).  It exists for callers that cannot allocate device memory when they
attend, e.g. code running inside a custom allocator."""
import ctypes

import pytest
import torch

import synthetic

pytestmark = [pytest.mark.gpu,
              pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA device")]


def test_noalloc_decode_matches_decode_twice():
    import block_sparse_attention_gb300 as bsa
    lib = bsa.load()
    f = lib.bsattn_decode_varlen_noalloc
    P, I = ctypes.c_void_p, ctypes.c_int
    f.argtypes = [P, P, P, P, P, I, P, I, I, I, I, I, I, I, P]
    f.restype = I

    dev = torch.device("cuda", torch.cuda.current_device())
    B, Hq, Hkv, d, Smax, nsel = 4, 16, 4, 128, 4096, 16
    sl, idx = synthetic.decode_selection(B, Hkv, 1000, Smax, nsel, nsel, seed=3)
    q, k, v = synthetic.decode_qkv(B, Hq, Hkv, Smax, d, torch.bfloat16, sl, seed=3)
    q, k, v, sl, idx = (t.to(dev) for t in (q, k, v, sl, idx))
    ns = 4
    want = bsa.bsattn_decode_varlen(q, k, v, sl, idx, ns)
    stream = torch.cuda.current_stream(dev).cuda_stream
    for _ in range(2):
        out = torch.full_like(q, float("nan"))
        rc = f(q.data_ptr(), k.data_ptr(), v.data_ptr(), sl.data_ptr(), idx.data_ptr(), ns,
               out.data_ptr(), B, Hq, Hkv, Smax, d, nsel, 1, stream)
        assert rc == 0, bsa.bsattn_status_string(rc)
        torch.cuda.synchronize()
        assert float((out.float() - want.float()).abs().max()) <= 2e-2

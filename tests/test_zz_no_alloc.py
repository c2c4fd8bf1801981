"""fia_decode_no_alloc: the decode entry point for callers that cannot allocate
device memory (it takes its scratch from an array built into the library).

Called through the C ABI with only input and output buffers, it must give the
same result as fia_decode with a caller workspace, on two calls in a row (the
second call reuses the scratch the first one left behind).  This file sorts
last so that a run stopping at its first failure has already run every other
test."""
import ctypes

import numpy as np
import pytest
import torch

import fia_inputs
from attention_fia_prefill_gb300 import _binding as B
from tests.parity import OUT_TOL, LSE_REL

pytestmark = pytest.mark.gpu


def _call_no_alloc(lib, c, dev, out, lse):
    prm = B.Params(num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                   input_layout="BNSD", actual_seq_kvlen=c.kv_lens, block_size=c.block_size, softmax_lse_flag=True)
    q, kp, vp, tb = (t.to(dev) for t in (c.q, c.k_pool, c.v_pool, c.block_table))
    d = [B.tensor_desc(t) for t in (q, kp, vp, tb, out, lse)]
    st = lib.fia_decode_no_alloc(ctypes.byref(d[0]), ctypes.byref(d[1]), ctypes.byref(d[2]), None, None,
                                 ctypes.byref(d[3]), None, ctypes.byref(prm.p), ctypes.byref(d[4]),
                                 ctypes.byref(d[5]), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st


def test_no_alloc_matches_fia_decode_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fia_prefill_gb300 as fia
    lib = B.load_library()
    dev = torch.device("cuda", 0)
    cases = [fia_inputs.paged_decode_case(5, 16, 4, 128, [4000, 3, 1200, 128, 2049], workload=7100),
             fia_inputs.workload_paged_gqa_decode()]
    for c in cases:
        ref_o, ref_l = fia.fia_decode(c.q.to(dev), c.k_pool.to(dev), c.v_pool.to(dev),
                                      block_table=c.block_table.to(dev), block_size=c.block_size,
                                      actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads,
                                      num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                      input_layout="BNSD", softmax_lse_flag=True)
        torch.cuda.synchronize()
        for _ in range(2):
            out = torch.full_like(ref_o, float("nan"))
            lse = torch.full_like(ref_l, float("nan"))
            st = _call_no_alloc(lib, c, dev, out, lse)
            assert st == 0, lib.fia_last_error().decode()
            err = (out.float() - ref_o.float()).abs().max().item()
            assert err <= OUT_TOL[torch.bfloat16], err
            lerr = ((lse - ref_l).abs() / ref_l.abs().clamp_min(1.0)).max().item()
            assert lerr <= LSE_REL, lerr


def _mla_no_alloc(lib, c, dev, out, lse):
    prm = B.Params(num_heads=c.num_heads, num_key_value_heads=1, scale_value=c.scale, input_layout="BSND",
                   actual_seq_kvlen=c.kv_lens, block_size=c.block_size, softmax_lse_flag=lse is not None)
    q, qr, lat, rope, tb = (t.to(dev) for t in (c.q, c.q_rope, c.latent, c.rope, c.block_table))
    d = [B.tensor_desc(t) for t in (q, lat, qr, rope, tb, out, lse)]
    st = lib.fia_decode_no_alloc(ctypes.byref(d[0]), ctypes.byref(d[1]), ctypes.byref(d[1]), ctypes.byref(d[2]),
                                 ctypes.byref(d[3]), ctypes.byref(d[4]), None, ctypes.byref(prm.p),
                                 ctypes.byref(d[5]), ctypes.byref(d[6]) if d[6] is not None else None,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return st


def test_no_alloc_mla_matches_fia_decode_twice():
    """The MLA branch (latent key = value, rope part) through the shared array,
    twice in a row, equals fia_decode with a caller workspace."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import attention_fia_prefill_gb300 as fia
    lib = B.load_library()
    dev = torch.device("cuda", 0)
    c = fia_inputs.mla_decode_case(3, 16, [700, 33, 2100], workload=7200)
    lat = c.latent.to(dev)
    ref_o, ref_l = fia.fia_decode(c.q.to(dev), lat, lat, query_rope=c.q_rope.to(dev), key_rope=c.rope.to(dev),
                                  block_table=c.block_table.to(dev), block_size=c.block_size,
                                  actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads, num_key_value_heads=1,
                                  scale_value=c.scale, input_layout="BSND", softmax_lse_flag=True)
    torch.cuda.synchronize()
    for _ in range(2):
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        st = _mla_no_alloc(lib, c, dev, out, lse)
        assert st == 0, lib.fia_last_error().decode()
        err = (out.float() - ref_o.float()).abs().max().item()
        assert err <= OUT_TOL[torch.bfloat16], err
        lerr = ((lse - ref_l).abs() / ref_l.abs().clamp_min(1.0)).max().item()
        assert lerr <= LSE_REL, lerr


def test_no_alloc_refuses_full_mla_workload():
    """MLA decode with 128 query heads (B=32, latent 512 + rope 64, length
    8192) needs more scratch than the built-in array holds: refused with
    FIA_ERR_WORKSPACE before any device work."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = B.load_library()
    P = 1 << 20
    q = B.raw_desc(P, B.DTYPE_BF16, (32, 1, 128, 512))
    qr = B.raw_desc(P, B.DTYPE_BF16, (32, 1, 128, 64))
    lat = B.raw_desc(P, B.DTYPE_BF16, (2048, 128, 512))
    rope = B.raw_desc(P, B.DTYPE_BF16, (2048, 128, 64))
    table = B.raw_desc(P, B.DTYPE_I32, (32, 64))
    prm = B.Params(num_heads=128, num_key_value_heads=1, input_layout="BSND", block_size=128,
                   actual_seq_kvlen=[8192])
    st = lib.fia_decode_no_alloc(ctypes.byref(q), ctypes.byref(lat), ctypes.byref(lat), ctypes.byref(qr),
                                 ctypes.byref(rope), ctypes.byref(table), None, ctypes.byref(prm.p), ctypes.byref(q),
                                 None, None)
    assert st == 8, lib.fia_last_error().decode()
    assert b"built-in maximum" in lib.fia_last_error()


def test_no_alloc_rejects_oversized_call():
    """A call whose scratch need exceeds the built-in maximum is refused before
    any device work (here: 4096 batches x 8 KV heads of split partials)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    lib = B.load_library()
    P = 1 << 20
    q = B.raw_desc(P, B.DTYPE_BF16, (4096, 32, 1, 128))
    pool = B.raw_desc(P, B.DTYPE_BF16, (40960, 8, 128, 128))
    table = B.raw_desc(P, B.DTYPE_I32, (4096, 10))
    prm = B.Params(num_heads=32, num_key_value_heads=8, input_layout="BNSD", block_size=128,
                   actual_seq_kvlen=[1000])
    st = lib.fia_decode_no_alloc(ctypes.byref(q), ctypes.byref(pool), ctypes.byref(pool), None, None,
                                 ctypes.byref(table), None, ctypes.byref(prm.p), ctypes.byref(q), None, None)
    assert st == 8
    assert b"built-in maximum" in lib.fia_last_error()

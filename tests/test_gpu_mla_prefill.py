"""MLA prefill (scores over 192 columns: query/key D 192, or D 128 plus
64-wide rope tensors; value D 128): the CUDA path through the C ABI against
the oracle on the same seeded inputs."""
import pytest
import torch

import fia_inputs
from oracle import fia_oracle
from tests.parity import assert_lse_close, assert_out_close, assert_rows_close

pytestmark = pytest.mark.gpu

INT32_MAX = 2147483647


def _run(fia, c, mode, pre=INT32_MAX, nxt=INT32_MAX):
    cuda = lambda x: None if x is None else x.cuda()
    out, lse = fia.fia_prefill_mla(c.q.cuda(), c.k.cuda(), c.v.cuda(), query_rope=cuda(c.q_rope),
                                   key_rope=cuda(c.k_rope), num_heads=c.num_heads,
                                   num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                   input_layout=c.layout, sparse_mode=mode, pre_tokens=pre, next_tokens=nxt,
                                   actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                                   softmax_lse_flag=True)
    torch.cuda.synchronize()
    return out, lse


def _oracle(c, mode, pre=INT32_MAX, nxt=INT32_MAX, rows=None):
    return fia_oracle.fia_prefill(c.q, c.k, c.v, query_rope=c.q_rope, key_rope=c.k_rope, num_heads=c.num_heads,
                                  num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                  input_layout=c.layout, sparse_mode=mode, pre_tokens=pre, next_tokens=nxt,
                                  actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen, rows=rows)


def _check(fia, c, mode, **kw):
    out, lse = _run(fia, c, mode, **kw)
    ref_o, ref_l = _oracle(c, mode, **kw)
    assert out.shape[-1] == (128 * c.num_heads if c.layout == "BSH" else 128)
    assert_out_close(out, ref_o, c.q.dtype)
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("rope,dtype,N1,N2", [(True, "bf16", 8, 2), (False, "f16", 4, 4)])
def test_mla_prefill_tnd_varlen(fia, rope, dtype, N1, N2):
    """TND, right-down causal: an empty sequence, 1-row and ragged sequences,
    a sequence spanning several pairs; both input forms."""
    lens = [1, 127, 300, 0, 700, 129]
    c = fia_inputs.mla_prefill_case(lens, lens, N1, N2, rope=rope, dtype=dtype, layout="TND",
                                    workload=4000 + N1 + int(rope))
    _check(fia, c, 3)


@pytest.mark.parametrize("layout,rope,mode", [("BNSD", False, 0), ("BSND", True, 2), ("BSH", True, 4)])
def test_mla_prefill_padded_layouts(fia, layout, rope, mode):
    """Padded layouts with unequal query / key lengths: no mask, left-up causal
    and a band (pre 100, next 20)."""
    c = fia_inputs.mla_prefill_case([300, 129], [260, 400], 4, 2, rope=rope, layout=layout,
                                    workload=4100 + mode)
    kw = {"pre": 100, "nxt": 20} if mode == 4 else {}
    _check(fia, c, mode, **kw)


def test_mla_prefill_forms_agree(fia):
    """Rope tensors and the same columns inside 192-wide query / key give the
    same bits (the kernel sees the same shared-memory tiles)."""
    c = fia_inputs.mla_prefill_case([500, 256], [500, 256], 4, 2, rope=True, layout="TND", workload=4200)
    out_r, lse_r = _run(fia, c, 3)
    c.q = torch.cat([c.q, c.q_rope], dim=-1).contiguous()
    c.k = torch.cat([c.k, c.k_rope], dim=-1).contiguous()
    c.q_rope = c.k_rope = None
    out_c, lse_c = _run(fia, c, 3)
    assert torch.equal(out_r, out_c) and torch.equal(lse_r, lse_c)


def test_mla_prefill_workload_sampled(fia):
    """The MLA prefill workload (8 sequences U[256,4096], 32 heads, 192 / 128):
    sampled rows against the oracle, first / last rows and tile edges."""
    c = fia_inputs.workload_mla_prefill()
    out, lse = _run(fia, c, 3)
    starts = [0] + c.actual_seq_qlen[:-1]
    rows = []
    for b, (s0, s1) in enumerate(zip(starts, c.actual_seq_qlen)):
        L = s1 - s0
        for h in (0, 31):
            for i in sorted({0, min(255, L - 1), L - 1}):
                rows.append((b, h, i))
    ref = _oracle(c, 3, rows=rows)
    assert_rows_close(out, lse, rows, ref, lambda r: (starts[r[0]] + r[2], r[1]), c.q.dtype)

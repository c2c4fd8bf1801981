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


def _run(fia, c, mode, pre=INT32_MAX, nxt=INT32_MAX, mask=None):
    cuda = lambda x: None if x is None else x.cuda()
    out, lse = fia.fia_prefill_mla(c.q.cuda(), c.k.cuda(), c.v.cuda(), query_rope=cuda(c.q_rope),
                                   key_rope=cuda(c.k_rope), atten_mask=cuda(mask), num_heads=c.num_heads,
                                   num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                   input_layout=c.layout, sparse_mode=mode, pre_tokens=pre, next_tokens=nxt,
                                   actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                                   softmax_lse_flag=True)
    torch.cuda.synchronize()
    return out, lse


def _oracle(c, mode, pre=INT32_MAX, nxt=INT32_MAX, rows=None, mask=None):
    return fia_oracle.fia_prefill(c.q, c.k, c.v, query_rope=c.q_rope, key_rope=c.k_rope, atten_mask=mask,
                                  num_heads=c.num_heads,
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


# (mode, layout, rope, dtype, mask shape, mask dtype, kind, pre, next): q lengths 300 / 129, key
# lengths 260 / 400, so S1 = 300 and S2 = 400 (+ padding of the mask's key axis)
MLA_MASK_CASES = [
    (1, "BNSD", True, "bf16", (2, 300, 400), "u8", "random", None, None),
    (1, "BSND", False, "f16", (300, 416), "bool", "blocks", None, None),
    (0, "BSH", True, "bf16", (2, 1, 300, 401), "i8", "blocks", 100, 20),
    (0, "BNSD", False, "bf16", (1, 300, 400), "u8", "random", 0, 300),
]


@pytest.mark.parametrize("mode,layout,rope,dtype,mshape,mdtype,kind,pre,nxt", MLA_MASK_CASES)
def test_mla_prefill_explicit_mask(fia, mode, layout, rope, dtype, mshape, mdtype, kind, pre, nxt):
    """An explicit atten_mask with MLA prefill (sparse_mode 1, and 0 with the
    pre/next window): mask shapes and dtypes, ragged query and key tails,
    fully masked rows, both input forms, element by element."""
    c = fia_inputs.mla_prefill_case([300, 129], [260, 400], 4, 2, rope=rope, dtype=dtype, layout=layout,
                                    workload=4300 + mode + mshape[-1])
    mask = fia_inputs.atten_mask(mshape, kind, dtype=mdtype, workload=4400 + mshape[-1])
    kw = {} if pre is None else {"pre": pre, "nxt": nxt}
    out, lse = _run(fia, c, mode, mask=mask, **kw)
    ref_o, ref_l = _oracle(c, mode, mask=mask, **kw)
    assert_out_close(out, ref_o, c.q.dtype)
    assert_lse_close(lse, ref_l)


def test_mla_prefill_mask_tnd_and_causal_bits(fia):
    """TND with a per-sequence mask indexed by each sequence's own rows and
    keys, against the oracle; and a lower-triangular mask in sparse_mode 1
    gives the same bits as sparse_mode 2 (the masked tiles only add zeros)."""
    lens_q, lens_kv = [1, 127, 300, 0, 700, 129], [5, 127, 260, 3, 700, 200]
    c = fia_inputs.mla_prefill_case(lens_q, lens_kv, 8, 2, rope=True, layout="TND", workload=4500)
    mask = fia_inputs.atten_mask((6, 700, 704), "blocks", workload=4501)
    out, lse = _run(fia, c, 1, mask=mask)
    ref_o, ref_l = _oracle(c, 1, mask=mask)
    assert_out_close(out, ref_o, c.q.dtype)
    assert_lse_close(lse, ref_l)
    c2 = fia_inputs.mla_prefill_case([700, 300], [700, 300], 4, 4, rope=False, layout="BNSD", workload=4502)
    causal = fia_inputs.atten_mask((700, 704), "causal")
    out_m, lse_m = _run(fia, c2, 1, mask=causal)
    out_c, lse_c = _run(fia, c2, 2)
    assert torch.equal(out_m, out_c) and torch.equal(lse_m, lse_c)


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

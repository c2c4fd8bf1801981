"""Block-sparse attention parity through the C ABI against the fp64 oracle."""
import numpy as np
import pytest
import torch

import fia_inputs
from oracle import fia_oracle
from tests.parity import assert_lse_close, assert_out_close, assert_rows_close

pytestmark = pytest.mark.gpu


def _run(fia, c, **kw):
    out, lse = fia.bsa_forward(c.q.cuda(), c.k.cuda(), c.v.cuda(), c.mask.cuda(), c.block_shape,
                               num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                               scale_value=c.scale, input_layout=c.layout, softmax_lse_flag=True, **kw)
    torch.cuda.synchronize()
    return out, lse


def _oracle(c, rows=None):
    return fia_oracle.bsa_forward(c.q, c.k, c.v, c.mask, c.block_shape, num_heads=c.num_heads,
                                  num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                  input_layout=c.layout, rows=rows)


@pytest.mark.parametrize("S,X,Y,keep", [(384, 128, 128, 0.3), (300, 128, 128, 0.5), (640, 256, 128, 0.3),
                                        (520, 128, 256, 0.4)])
def test_small(fia, S, X, Y, keep):
    c = fia_inputs.bsa_case(1, 4, 2, S, S, 128, X=X, Y=Y, keep=keep, workload=3000 + S)
    out, lse = _run(fia, c)
    ro, rl = _oracle(c)
    assert_out_close(out, ro, torch.bfloat16)
    assert_lse_close(lse, rl)


def test_empty_rows_without_diagonal(fia):
    """Mask rows that keep no block give 0 / +inf."""
    c = fia_inputs.bsa_case(1, 2, 2, 256, 256, 64, keep=0.0, diagonal=False, dtype="f16", workload=3100)
    c.mask[0, 0, 1, 0] = 1
    out, lse = _run(fia, c)
    ro, rl = _oracle(c)
    assert_out_close(out, ro, torch.float16)
    assert_lse_close(lse, rl)


def test_all_ones_equals_dense(fia):
    c = fia_inputs.bsa_case(2, 4, 2, 300, 300, 128, keep=1.0, workload=3200)
    o1, l1 = _run(fia, c)
    o2, l2 = fia.fia_prefill(c.q.cuda(), c.k.cuda(), c.v.cuda(), num_heads=4, num_key_value_heads=2,
                             scale_value=c.scale, input_layout="BNSD", softmax_lse_flag=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_full_bsa_workload_sampled(fia):
    """Block-sparse prefill bf16: B=2, 32/8 heads, S=16384, D=128, 128x128
    blocks, diagonal + ~25% -- at full size, one row of every other work item
    (one query block of one head: 4096 rows, the first, last and a random row
    of the block in turn) vs the oracle."""
    c = fia_inputs.workload_bsa()
    out, lse = _run(fia, c)
    rng = np.random.default_rng(5)
    rows = []
    for b in range(2):
        for h in range(32):
            for qb in range((b + h) % 2, 128, 2):
                rows.append((b, h, qb * 128 + (0, 127, int(rng.integers(128)))[(h + qb) % 3]))
    ref = _oracle(c, rows=rows)
    assert_rows_close(out, lse, rows, ref, lambda r: (r[0], r[1], r[2]), torch.bfloat16)


# ------------------------------------------------------------ FP8
def _run_fp8(fia, f, **kw):
    c = f.base
    m = None if c.mask is None else c.mask.cuda()
    out, lse = fia.bsa_forward(c.q.cuda(), c.k.cuda(), c.v.cuda(), m, c.block_shape,
                               num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                               scale_value=c.scale, input_layout=c.layout, softmax_lse_flag=True,
                               actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.actual_seq_kvlen,
                               q_dequant_scale=f.q_scale.cuda(), k_dequant_scale=f.k_scale.cuda(),
                               v_dequant_scale=f.v_scale.cuda(), **kw)
    torch.cuda.synchronize()
    assert out.dtype == torch.bfloat16
    return out, lse


def _fp8_atol(f, ref_absmax):
    """Bound on |out - oracle| for the FP8 path, from its arithmetic: the
    scores are exact (e4m3 products, fp32 sums); V enters exactly (e4m3 in
    f16) and P times the value scale is rounded to f16 (2^-11 relative), so
    out moves by at most 2^-11 * max|V| (2^-10 taken); the bf16 output adds
    2^-9 * |out|; 2e-3 covers exp2 and fp32 sums.  Never below the bf16 bound."""
    v_max = float(f.base.v.float().abs().max()) * float(f.v_scale.max())
    return max(1.6e-2, 2.0 ** -9 * ref_absmax + 2.0 ** -10 * v_max + 2e-3)


def _assert_fp8_close(f, out, ref):
    ref = np.asarray(ref, dtype=np.float64)
    g = out.float().cpu().numpy().astype(np.float64)
    assert g.shape == ref.shape and np.all(np.isfinite(g))
    tol = _fp8_atol(f, float(np.abs(ref).max()))
    err = float(np.abs(g - ref).max())
    assert err <= tol, f"FP8 attention_out: max abs err {err:.3e} > {tol:.3e}"


def _oracle_fp8(f, rows=None):
    c = f.base
    return fia_oracle.bsa_forward(c.q, c.k, c.v, c.mask, c.block_shape, num_heads=c.num_heads,
                                  num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                  input_layout=c.layout, actual_seq_qlen=c.actual_seq_qlen,
                                  actual_seq_kvlen=c.actual_seq_kvlen, rows=rows, q_dequant_scale=f.q_scale,
                                  k_dequant_scale=f.k_scale, v_dequant_scale=f.v_scale)


@pytest.mark.parametrize("Sq,Skv,Y,layout", [(300, 600, 256, "BNSD"), (384, 1100, 512, "BNSD"),
                                             (257, 513, 256, "BSND")])
def test_fp8_small(fia, Sq, Skv, Y, layout):
    """FP8 e4m3 query/key/value with per-block dequant scales (128 query rows,
    Y key rows): ragged query and key tails, both quantisation block sizes,
    BNSD and BSND; the bf16 output within the bound the FP8 arithmetic
    gives (_fp8_atol) of the oracle on the dequantised values."""
    f = fia_inputs.bsa_fp8_case(2, 4, 2, Sq, Skv, Y, keep=0.4, workload=3500 + Sq + Y, layout=layout)
    out, lse = _run_fp8(fia, f)
    ro, rl = _oracle_fp8(f)
    _assert_fp8_close(f, out, ro)
    assert_lse_close(lse, rl)


def test_fp8_tnd_varlen(fia):
    """TND: per-sequence blocks of the scales and the mask, an empty sequence."""
    lens = [1, 300, 0, 513]
    T = sum(lens)
    f = fia_inputs.bsa_fp8_case(4, 4, 2, max(lens), max(lens), 256, keep=0.5, workload=3600)
    c = f.base
    c.q = fia_inputs.fp8_e4m3((T, 4, 128), 3600, 40)
    c.k = fia_inputs.fp8_e4m3((T, 2, 128), 3600, 41)
    c.v = fia_inputs.fp8_e4m3((T, 2, 128), 3600, 42)
    c.layout = "TND"
    c.actual_seq_qlen = c.actual_seq_kvlen = fia_inputs.cumsum_no_leading_zero(lens)
    out, lse = _run_fp8(fia, f)
    ro, rl = _oracle_fp8(f)
    _assert_fp8_close(f, out, ro)
    assert_lse_close(lse, rl)


def test_fp8_workload_sampled(fia):
    """FP8 block-sparse workload (B=2, 32/8 heads, S=16384, 128 x 256 blocks,
    diagonal + ~25%): sampled rows against the oracle."""
    f = fia_inputs.workload_bsa_fp8()
    out, lse = _run_fp8(fia, f)
    rows = [(b, h, i) for b in (0, 1) for h in (0, 17, 31) for i in (0, 127, 128, 8191, 16383)]
    ref = _oracle_fp8(f, rows=rows)
    got = torch.stack([out[b, h, i] for (b, h, i) in rows])
    _assert_fp8_close(f, got, np.stack([o for o, _ in ref]))
    for (b, h, i), (_, l_ref) in zip(rows, ref):
        assert abs(float(lse[b, h, i, 0]) - l_ref) <= 1e-3 * max(1.0, abs(l_ref)), (b, h, i)


def test_fp8_dense_without_mask(fia):
    """FP8 prefill without a block mask (every block kept, dense attention):
    against the oracle with an all-ones mask, and the same bits as the call
    given that all-ones mask."""
    f = fia_inputs.bsa_fp8_case(2, 4, 2, 300, 600, 256, keep=0.4, workload=3650)
    f.base.mask = torch.ones_like(f.base.mask)
    out_m, lse_m = _run_fp8(fia, f)
    ro, rl = _oracle_fp8(f)
    _assert_fp8_close(f, out_m, ro)
    assert_lse_close(lse_m, rl)
    mask = f.base.mask
    f.base.mask = None
    try:
        out_n, lse_n = _run_fp8(fia, f)
    finally:
        f.base.mask = mask
    assert torch.equal(out_m, out_n) and torch.equal(lse_m, lse_n)


@pytest.mark.parametrize("which", ["q", "k", "v"])
def test_fp8_nonpositive_scale_reported(fia, which):
    """A dequant scale that is not positive (BSA "FP8特性说明": the scales
    describe what each block is worth) makes the call report
    FIA_ERR_UNSUPPORTED through the device status word; a call with valid
    scales on the same workspace afterwards reports FIA_OK."""
    f = fia_inputs.bsa_fp8_case(1, 2, 1, 256, 512, 256, keep=1.0, workload=3600)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device="cuda")
    bad = {"q": f.q_scale.clone(), "k": f.k_scale.clone(), "v": f.v_scale.clone()}
    bad[which].view(-1)[0] = -1.0 if which != "v" else 0.0
    c = f.base
    dev = "cuda"
    fia.bsa_forward(c.q.to(dev), c.k.to(dev), c.v.to(dev), c.mask.to(dev), c.block_shape, num_heads=c.num_heads,
                    num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
                    workspace=ws, q_dequant_scale=bad["q"].to(dev), k_dequant_scale=bad["k"].to(dev),
                    v_dequant_scale=bad["v"].to(dev))
    assert fia.fia_device_status(ws) == 5
    _run_fp8(fia, f, workspace=ws)
    assert fia.fia_device_status(ws) == 0

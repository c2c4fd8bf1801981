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
    blocks, diagonal + ~25% -- at full size, sampled rows vs the oracle."""
    c = fia_inputs.workload_bsa()
    out, lse = _run(fia, c)
    rng = np.random.default_rng(5)
    rows = [(int(rng.integers(2)), int(rng.integers(32)), int(i)) for i in
            [0, 1, 127, 128, 8191, 16383] + list(rng.integers(16384, size=10))]
    ref = _oracle(c, rows=rows)
    assert_rows_close(out, lse, rows, ref, lambda r: (r[0], r[1], r[2]), torch.bfloat16)

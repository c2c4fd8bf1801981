"""MLA decode parity (npu_fused_infer_attention_score_v2 with query_rope /
key_rope): key = value = the 512-d latent cache, scores add the 64-d rope
part, one kv head for every query head.  Checked through the C ABI against
the fp64 oracle; poisoned caches (NaN block behind unused table entries, NaN
rows past each sequence) expose any read outside a sequence."""
import numpy as np
import pytest
import torch

import fia_inputs
from tests import parity
from oracle import fia_oracle
from tests.parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


def _run(fia, c, **kw):
    dev = "cuda"
    lat = c.latent.to(dev)
    out, lse = fia.fia_decode(c.q.to(dev), lat, lat, query_rope=c.q_rope.to(dev), key_rope=c.rope.to(dev),
                              block_table=c.block_table.to(dev), block_size=c.block_size,
                              actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads, num_key_value_heads=1,
                              scale_value=c.scale, input_layout="BSND", softmax_lse_flag=True, **kw)
    torch.cuda.synchronize()
    return out, lse


def _oracle(c, rows=None):
    return fia_oracle.fia_decode(c.q, c.latent, c.latent, num_heads=c.num_heads, num_key_value_heads=1,
                                 scale_value=c.scale, input_layout="BSND", actual_seq_kvlen=c.kv_lens,
                                 block_table=c.block_table, block_size=c.block_size, query_rope=c.q_rope,
                                 key_rope=c.rope, rows=rows)


def _check(fia, c):
    out, lse = _run(fia, c)
    ro, rl = _oracle(c)
    assert_out_close(out, ro, c.q.dtype)
    assert_lse_close(lse, rl)
    return out, lse


def test_mla_small_ragged(fia):
    """16 heads, lengths spanning one token, several 32-token stages and a ragged tail."""
    _check(fia, fia_inputs.mla_decode_case(3, 16, [1, 100, 300], workload=4100, poison=True))


def test_mla_128_heads(fia):
    _check(fia, fia_inputs.mla_decode_case(2, 128, [2049, 31], workload=4200, poison=True))


def test_mla_block_size_16(fia):
    """Pages of 16 tokens: each 32-key stage gathers two pages."""
    _check(fia, fia_inputs.mla_decode_case(2, 32, [77, 200], block_size=16, workload=4300, poison=True))


def test_mla_empty_sequence(fia):
    """kv length 0: attention_out = 0 and softmax_lse = +inf for that batch."""
    c = fia_inputs.mla_decode_case(3, 16, [0, 50, 0], workload=4400, poison=True)
    out, lse = _check(fia, c)
    assert torch.all(out[0] == 0) and torch.all(out[2] == 0)
    assert torch.all(torch.isinf(lse[0])) and torch.all(lse[0] > 0)


def test_mla_full_workload(fia):
    """MLA decode bf16: B=32, 128 heads, kv length 8192 per batch, block 128 --
    every output finite, 8 heads of every batch (256 rows, each batch's
    segments and merge) against the oracle."""
    c = fia_inputs.workload_mla_decode()
    out, lse = _run(fia, c)
    assert torch.isfinite(out.float()).all()
    rng = np.random.default_rng(5)
    rows = [(b, h) for b in range(32) for h in sorted(rng.choice(128, 8, replace=False).tolist())]
    pairs = _oracle(c, rows=rows)
    worst = worst_lse = 0.0
    for (b, h), (ro, rl) in zip(rows, pairs):
        got = out[b, 0, h].float().cpu().numpy()
        err = float(np.abs(got - ro).max())
        rel = abs(float(lse[b, h, 0, 0]) - rl) / max(1.0, abs(rl))
        worst, worst_lse = max(worst, err), max(worst_lse, rel)
        assert err <= 1.6e-2, (b, h, err)
        assert rel <= 1e-3, (b, h)
    parity._record("sampled rows max abs", worst)
    parity._record("sampled rows lse max rel", worst_lse)

"""Prefill against a paged KV cache (chunked prefill): the CUDA path through
the C ABI against the oracle's paged prefill on the same seeded inputs.  The
pools hide NaN behind unused table entries and past each sequence's keys."""
import pytest
import torch

import fia_inputs
from oracle import fia_oracle
from tests.parity import assert_lse_close, assert_out_close, assert_rows_close

pytestmark = pytest.mark.gpu

INT32_MAX = 2147483647


def _run(fia, c, mode, mask=None, pre=INT32_MAX, nxt=INT32_MAX):
    out, lse = fia.fia_prefill_paged(c.q.cuda(), c.k_pool.cuda(), c.v_pool.cuda(), c.block_table.cuda(),
                                     block_size=c.block_size, actual_seq_kvlen=c.kv_lens,
                                     actual_seq_qlen=c.actual_seq_qlen, num_heads=c.num_heads,
                                     num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                     input_layout=c.layout, sparse_mode=mode, pre_tokens=pre, next_tokens=nxt,
                                     atten_mask=None if mask is None else mask.cuda(), softmax_lse_flag=True)
    torch.cuda.synchronize()
    return out, lse


def _oracle(c, mode, mask=None, pre=INT32_MAX, nxt=INT32_MAX, rows=None):
    return fia_oracle.fia_prefill_paged(c.q, c.k_pool, c.v_pool, block_table=c.block_table,
                                        block_size=c.block_size, actual_seq_kvlen=c.kv_lens,
                                        num_heads=c.num_heads, num_key_value_heads=c.num_key_value_heads,
                                        input_layout=c.layout, scale_value=c.scale, sparse_mode=mode,
                                        actual_seq_qlen=c.actual_seq_qlen, atten_mask=mask, pre_tokens=pre,
                                        next_tokens=nxt, rows=rows)


def _check(fia, c, mode, **kw):
    out, lse = _run(fia, c, mode, **kw)
    ref_o, ref_l = _oracle(c, mode, **kw)
    assert_out_close(out, ref_o, c.q.dtype)
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("bs,layout_kv,D,dtype,mode,layout", [
    (128, "BNBD", 128, "bf16", 3, "BNSD"),
    (256, "BBH", 64, "f16", 3, "BSND"),
    (512, "BNBD", 128, "f16", 0, "BSH"),
    (384, "BBH", 128, "bf16", 2, "BNSD"),
])
def test_paged_prefill_chunks(fia, bs, layout_kv, D, dtype, mode, layout):
    """Chunks of 300 / 128 / 77 new rows after 700 / 0 / 1500 cached keys:
    every block size the pages allow, both pool layouts, ragged last blocks."""
    c = fia_inputs.paged_prefill_case([300, 128, 77], [1000, 128, 1577], 8, 2, D, bs, dtype, layout, layout_kv,
                                      workload=3000 + bs + D + mode)
    _check(fia, c, mode)


def test_paged_prefill_tnd(fia):
    """TND query (cumulative actual_seq_qlen) with per-sequence key counts,
    including an empty chunk and a chunk longer than its cache context."""
    c = fia_inputs.paged_prefill_case([1, 200, 0, 333], [50, 200, 7, 900], 8, 2, 128, 256, "bf16", "TND", "BNBD",
                                      workload=3100)
    _check(fia, c, 3)


def test_paged_prefill_band_and_mask(fia):
    """The band (sparse_mode 4) and an explicit mask (sparse_mode 1) over paged keys."""
    c = fia_inputs.paged_prefill_case([300, 260], [900, 260], 4, 2, 128, 128, "bf16", "BNSD", "BBH", workload=3200)
    _check(fia, c, 4, pre=300, nxt=0)
    mask = fia_inputs.atten_mask((2, 300, 912), "blocks", workload=3201)
    _check(fia, c, 1, mask=mask)


def test_paged_prefill_matches_contiguous(fia):
    """The same keys paged or contiguous give the same bits (only the K/V tile
    addresses differ)."""
    c = fia_inputs.paged_prefill_case([256, 200], [700, 333], 8, 2, 128, 256, "bf16", "BNSD", "BNBD", workload=3300)
    out_p, lse_p = _run(fia, c, 3)
    S = max(c.kv_lens)
    k = torch.zeros((2, 2, S, 128), dtype=torch.bfloat16)
    v = torch.zeros_like(k)
    for b, L in enumerate(c.kv_lens):
        for j in range(L):
            blk = int(c.block_table[b, j // c.block_size])
            k[b, :, j] = c.k_pool[blk, :, j % c.block_size]
            v[b, :, j] = c.v_pool[blk, :, j % c.block_size]
    out_c, lse_c = fia.fia_prefill(c.q.cuda(), k.cuda(), v.cuda(), num_heads=8, num_key_value_heads=2,
                                   scale_value=c.scale, input_layout="BNSD", sparse_mode=3,
                                   actual_seq_qlen=c.actual_seq_qlen, actual_seq_kvlen=c.kv_lens,
                                   softmax_lse_flag=True)
    torch.cuda.synchronize()
    assert torch.equal(out_p, out_c) and torch.equal(lse_p, lse_c)


def test_chunked_prefill_workload_sampled(fia):
    """The chunked-prefill workload (8 x 2048-token chunks after cached contexts
    U[0, 14336], 32/8 heads, 256-token blocks): 512 sampled rows against the
    oracle, one of every (sequence, 256-row item, kv group)."""
    c = fia_inputs.workload_chunked_prefill()
    out, lse = _run(fia, c, 3)
    # one row of every (sequence, 256-row item, kv group): its head cycling
    # through the group, its position over the two tiles' edges
    rows = []
    for b in range(len(c.kv_lens)):
        for q0 in range(0, 2048, 256):
            for grp in range(8):
                k = q0 // 256 + grp
                rows.append((b, 4 * grp + k % 4, q0 + (0, 127, 128, 255)[k % 4]))
    ref = _oracle(c, 3, rows=rows)
    assert_rows_close(out, lse, rows, ref, lambda r: (r[0], r[1], r[2]), c.q.dtype)

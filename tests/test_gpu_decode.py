"""Decode parity: paged / contiguous incremental attention through the C ABI
against the fp64 oracle.  Pools carry a NaN block that unused block_table
entries point to, and NaN rows past each sequence's length, so any read
outside the sequence shows up as a non-finite output."""
import numpy as np
import pytest
import torch

import fia_inputs
from oracle import fia_oracle
from tests.parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


def _run_paged(fia, c, **kw):
    dev = "cuda"
    out, lse = fia.fia_decode(c.q.to(dev), c.k_pool.to(dev), c.v_pool.to(dev), block_table=c.block_table.to(dev),
                              block_size=c.block_size, actual_seq_kvlen=c.kv_lens, num_heads=c.num_heads,
                              num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
                              softmax_lse_flag=True, **kw)
    torch.cuda.synchronize()
    return out, lse


def _oracle_paged(c):
    return fia_oracle.fia_decode(c.q, c.k_pool, c.v_pool, num_heads=c.num_heads,
                                 num_key_value_heads=c.num_key_value_heads, scale_value=c.scale, input_layout="BNSD",
                                 actual_seq_kvlen=c.kv_lens, block_table=c.block_table, block_size=c.block_size)


def _check_paged(fia, c):
    out, lse = _run_paged(fia, c)
    ro, rl = _oracle_paged(c)
    assert_out_close(out, ro, c.q.dtype)
    assert_lse_close(lse, rl)
    return out, lse


def test_full_paged_gqa_workload(fia):
    """Decode GQA bf16 with paged KV: B=16, Q_N=32, KV_N=8, D=128, lengths
    uniform on [1, 4096], block 128, random physical blocks -- every output."""
    _check_paged(fia, fia_inputs.workload_paged_gqa_decode())


@pytest.mark.parametrize("bs", [16, 64, 128, 256])
def test_block_sizes(fia, bs):
    lens = [1, 15, 16, 17, 300, 0, 513]
    c = fia_inputs.paged_decode_case(len(lens), 8, 2, 128, lens, block_size=bs, workload=2000 + bs)
    _check_paged(fia, c)


@pytest.mark.parametrize("n1,n2", [(4, 4), (6, 3), (6, 2), (16, 2), (24, 1), (40, 1), (64, 1), (128, 2)])
def test_group_sizes(fia, n1, n2):
    """Head groups 1..64: a group's heads are the rows of one query tile (four
    copies up to 32 heads, two copies above)."""
    c = fia_inputs.paged_decode_case(3, n1, n2, 128, [200, 1, 129], block_size=128, workload=2100 + n1)
    _check_paged(fia, c)


@pytest.mark.parametrize("dtype,D", [("f16", 128), ("bf16", 64), ("f16", 64)])
def test_dtypes_and_head_dim(fia, dtype, D):
    c = fia_inputs.paged_decode_case(4, 8, 2, D, [77, 128, 1000, 3], block_size=128, dtype=dtype, workload=2200 + D)
    _check_paged(fia, c)


def test_bsh_cache_layout(fia):
    """(blocknum, block_size, KV_N * D) cache layout."""
    c = fia_inputs.paged_decode_case(3, 8, 4, 128, [300, 20, 129], block_size=128, workload=2300, layout_kv="BSH")
    _check_paged(fia, c)


def test_contiguous_bnsd(fia):
    """Non-paged decode: K/V (B, N2, S, D) with per-batch actual lengths."""
    B, N1, N2, S, D = 3, 8, 2, 700, 128
    q = fia_inputs.normal((B, N1, 1, D), "bf16", 2400, 1)
    k = fia_inputs.normal((B, N2, S, D), "bf16", 2400, 2)
    v = fia_inputs.normal((B, N2, S, D), "bf16", 2400, 3)
    lens = [700, 1, 333]
    out, lse = fia.fia_decode(q.cuda(), k.cuda(), v.cuda(), actual_seq_kvlen=lens, num_heads=N1,
                              num_key_value_heads=N2, scale_value=D ** -0.5, input_layout="BNSD",
                              softmax_lse_flag=True)
    torch.cuda.synchronize()
    ro, rl = fia_oracle.fia_decode(q, k, v, num_heads=N1, num_key_value_heads=N2, scale_value=D ** -0.5,
                                   input_layout="BNSD", actual_seq_kvlen=lens)
    assert_out_close(out, ro, torch.bfloat16)
    assert_lse_close(lse, rl)


def test_contiguous_bsnd(fia):
    B, N1, N2, S, D = 2, 4, 4, 260, 64
    q = fia_inputs.normal((B, 1, N1, D), "f16", 2500, 1)
    k = fia_inputs.normal((B, S, N2, D), "f16", 2500, 2)
    v = fia_inputs.normal((B, S, N2, D), "f16", 2500, 3)
    out, lse = fia.fia_decode(q.cuda(), k.cuda(), v.cuda(), num_heads=N1, scale_value=0.1, input_layout="BSND",
                              softmax_lse_flag=True)
    torch.cuda.synchronize()
    ro, rl = fia_oracle.fia_decode(q, k, v, num_heads=N1, scale_value=0.1, input_layout="BSND")
    assert_out_close(out, ro, torch.float16)
    assert_lse_close(lse, rl)


def test_paged_equals_contiguous_bitwise(fia):
    """The same cache read through a block_table or contiguously gives the
    same bits (same kernel arithmetic, only the addressing differs)."""
    B, N1, N2, S, D, bs = 2, 8, 2, 512, 128, 128
    k = fia_inputs.normal((B, N2, S, D), "bf16", 2600, 2)
    v = fia_inputs.normal((B, N2, S, D), "bf16", 2600, 3)
    q = fia_inputs.normal((B, N1, 1, D), "bf16", 2600, 1)
    lens = [512, 300]
    nb = S // bs
    perm = np.random.default_rng(1).permutation(B * nb)
    table = torch.from_numpy(perm.reshape(B, nb).astype(np.int32))
    kp = torch.empty((B * nb, N2, bs, D), dtype=torch.bfloat16)
    vp = torch.empty_like(kp)
    for b in range(B):
        for i in range(nb):
            kp[table[b, i]] = k[b, :, i * bs:(i + 1) * bs]
            vp[table[b, i]] = v[b, :, i * bs:(i + 1) * bs]
    o1, l1 = fia.fia_decode(q.cuda(), k.cuda(), v.cuda(), actual_seq_kvlen=lens, num_heads=N1, num_key_value_heads=N2,
                            scale_value=0.088, input_layout="BNSD", softmax_lse_flag=True)
    o2, l2 = fia.fia_decode(q.cuda(), kp.cuda(), vp.cuda(), block_table=table.cuda(), block_size=bs,
                            actual_seq_kvlen=lens, num_heads=N1, num_key_value_heads=N2, scale_value=0.088,
                            input_layout="BNSD", softmax_lse_flag=True)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_all_lengths_zero(fia):
    c = fia_inputs.paged_decode_case(2, 4, 2, 128, [0, 0], block_size=128, workload=2700)
    out, lse = _run_paged(fia, c)
    assert torch.all(out == 0) and torch.all(torch.isinf(lse) & (lse > 0))


def test_deterministic(fia):
    c = fia_inputs.paged_decode_case(5, 16, 4, 128, [4000, 3, 1200, 128, 2049], workload=2800)
    o1, l1 = _run_paged(fia, c)
    o2, l2 = _run_paged(fia, c)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_device_status_ok(fia):
    c = fia_inputs.paged_decode_case(2, 8, 2, 128, [100, 1000], workload=2900)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device="cuda")
    _run_paged(fia, c, workspace=ws)
    assert fia.fia_device_status(ws) == 0


def test_many_short_sequences(fia):
    """Many units with one or two stages each: CTAs cross many unit boundaries
    and merge partials of units they finish."""
    lens = [1, 130, 2, 257, 0, 5, 129, 128, 64, 1000, 3, 300] * 3
    c = fia_inputs.paged_decode_case(len(lens), 8, 2, 128, lens, block_size=128, workload=3000)
    _check_paged(fia, c)


@pytest.mark.gpu
def test_plan_in_workspace(fia):
    """A 160-batch plan (320 units, ~330 segments) read from the workspace."""
    rng = np.random.default_rng(77)
    lens = [int(x) for x in rng.integers(0, 300, size=160)]
    c = fia_inputs.paged_decode_case(len(lens), 8, 2, 128, lens, block_size=128, workload=3100)
    _check_paged(fia, c)


# ------------------------------------------------------- several query tokens
def _check_tokens(fia, c, mode):
    out, lse = _run_paged(fia, c, sparse_mode=mode)
    ro, rl = fia_oracle.fia_decode(c.q, c.k_pool, c.v_pool, num_heads=c.num_heads,
                                   num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                   input_layout="BNSD", actual_seq_kvlen=c.kv_lens, block_table=c.block_table,
                                   block_size=c.block_size, sparse_mode=mode)
    assert out.shape == c.q.shape and lse.shape == (c.q.shape[0], c.num_heads, c.q.shape[2], 1)
    assert_out_close(out, ro, c.q.dtype)
    assert_lse_close(lse, rl)


@pytest.mark.parametrize("qs", [2, 4, 8])
def test_query_tokens_causal(fia, qs):
    """Q_S new tokens per sequence, right-down causal (sparse_mode 3): token t
    sees the cache up to key S_kv - Q_S + t.  Lengths shorter than Q_S leave
    the first tokens without keys (0 / +inf)."""
    c = fia_inputs.paged_decode_case(4, 8, 2, 128, [300, 5, 1000, 129], block_size=64, workload=3200 + qs,
                                     q_tokens=qs)
    _check_tokens(fia, c, 3)


@pytest.mark.parametrize("mode,qs,D,n1,n2", [(0, 4, 128, 8, 2), (2, 3, 128, 4, 4), (3, 16, 64, 4, 1),
                                             (3, 2, 128, 32, 1)])
def test_query_tokens_modes(fia, mode, qs, D, n1, n2):
    """No mask, top-left causal, and the widest row count (64 = 4 heads x 16
    tokens, 32 heads x 2 tokens)."""
    c = fia_inputs.paged_decode_case(3, n1, n2, D, [700, 17, 2050], block_size=128, workload=3300 + mode + qs,
                                     q_tokens=qs)
    _check_tokens(fia, c, mode)


def test_query_tokens_full_workload_sampled(fia):
    """The headline paged workload (B=16, 32/8 heads, D=128, U[1,4096]) with
    4 new tokens per sequence, causal: sampled (batch, head) rows."""
    base = fia_inputs.workload_paged_gqa_decode()
    c = fia_inputs.paged_decode_case(16, 32, 8, 128, base.kv_lens, block_size=128, workload=3400, q_tokens=4)
    out, lse = _run_paged(fia, c, sparse_mode=3)
    rng = np.random.default_rng(9)
    rows = [(int(b), int(h)) for b, h in zip(rng.integers(16, size=12), rng.integers(32, size=12))] + [(15, 31)]
    ref = fia_oracle.fia_decode(c.q, c.k_pool, c.v_pool, num_heads=32, num_key_value_heads=8, scale_value=c.scale,
                                input_layout="BNSD", actual_seq_kvlen=c.kv_lens, block_table=c.block_table,
                                block_size=128, sparse_mode=3, rows=rows)
    for (b, h), (ro, rl) in zip(rows, ref):
        assert_out_close(out[b, h], torch.from_numpy(ro), c.q.dtype)
        assert_lse_close(lse[b, h, :, 0], torch.from_numpy(rl))


@pytest.mark.gpu
def test_plan_in_workspace_wide(fia):
    """A 700-batch plan (1400 units) is larger than the kernel parameters
    carry: it goes to the workspace as 32-bit words."""
    rng = np.random.default_rng(78)
    lens = [int(x) for x in rng.integers(0, 260, size=700)]
    c = fia_inputs.paged_decode_case(len(lens), 4, 2, 128, lens, block_size=128, workload=3150)
    _check_paged(fia, c)


def _check_rows(fia, c, rows, mode=0):
    out, lse = _run_paged(fia, c, sparse_mode=mode)
    ref = fia_oracle.fia_decode(c.q, c.k_pool, c.v_pool, num_heads=c.num_heads,
                                num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                input_layout="BNSD", actual_seq_kvlen=c.kv_lens, block_table=c.block_table,
                                block_size=c.block_size, sparse_mode=mode, rows=rows)
    for (b, h), (ro, rl) in zip(rows, ref):
        if c.q.shape[2] == 1:
            assert_out_close(out[b, h, 0], torch.from_numpy(ro), c.q.dtype)
            assert_lse_close(lse[b, h, 0, 0], torch.tensor(rl))
        else:
            assert_out_close(out[b, h], torch.from_numpy(ro), c.q.dtype)
            assert_lse_close(lse[b, h, :, 0], torch.from_numpy(rl))


@pytest.mark.parametrize("B,n1,n2,L,qs", [(8, 32, 8, 16384, 1), (16, 64, 1, 9000, 1), (16, 16, 1, 9000, 4)])
def test_long_segments_chunked(fia, B, n1, n2, L, qs):
    """Segments longer than the S^T tiles TMEM holds at once (31 stages for up
    to 16 rows, 7 for 64): the softmax runs chunk by chunk and rescales what
    earlier chunks of the segment accumulated.  Sampled (batch, head) rows,
    every row of batch 0's first kv head included."""
    c = fia_inputs.paged_decode_case(B, n1, n2, 128, [L] * B, block_size=128, workload=3500 + n1 + qs,
                                     q_tokens=qs)
    rng = np.random.default_rng(n1)
    rows = [(0, h) for h in range(n1 // n2)]
    rows += [(int(b), int(h)) for b, h in zip(rng.integers(B, size=10), rng.integers(n1, size=10))]
    _check_rows(fia, c, rows, mode=3 if qs > 1 else 0)


def test_device_timeout_path(fia):
    """The device-side failure path (the pages' "aicore timeout"): with a
    test-only wait limit of 1 ns every kernel wait that can give up does so,
    the call's status word reads FIA_ERR_TIMEOUT, and a normal call on the
    same stream and workspace afterwards succeeds with the right result."""
    from attention_fia_prefill_gb300 import _binding as B
    lib = B.load_library()
    c = fia_inputs.paged_decode_case(4, 8, 2, 128, [3000, 2000, 4000, 100], workload=3600)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device="cuda")
    lib.fia_debug_set_wait_limit_ns(1)
    try:
        _run_paged(fia, c, workspace=ws)
        status = fia.fia_device_status(ws)
    finally:
        lib.fia_debug_set_wait_limit_ns(0)
    assert status == 10, status
    out, lse = _run_paged(fia, c, workspace=ws)
    assert fia.fia_device_status(ws) == 0
    ro, rl = _oracle_paged(c)
    assert_out_close(out, ro, c.q.dtype)
    assert_lse_close(lse, rl)


@pytest.fixture(params=[0, 1], ids=["warp_mma", "tensor_core"])
def decode_path(request):
    """Both kernels that can serve units of at most 16 rows (head_dim 128):
    the warp-level mma.sync one (the default) and the tcgen05 one of larger
    units."""
    from attention_fia_prefill_gb300 import _binding as B
    lib = B.load_library()
    lib.fia_debug_set_decode_path(request.param)
    yield request.param
    lib.fia_debug_set_decode_path(0)


@pytest.mark.parametrize("n1,n2,qs,mode,bs", [(8, 2, 1, 0, 128), (4, 4, 1, 0, 16), (6, 2, 1, 0, 64),
                                              (4, 2, 1, 0, 256), (4, 2, 2, 3, 64), (1, 1, 4, 3, 128),
                                              (2, 1, 2, 2, 128), (3, 1, 1, 0, 16), (16, 2, 1, 0, 128),
                                              (8, 1, 1, 0, 64), (8, 2, 4, 3, 128), (6, 1, 2, 2, 16),
                                              (5, 1, 3, 3, 256), (32, 2, 1, 0, 128)])
def test_small_units_both_paths(fia, decode_path, n1, n2, qs, mode, bs):
    """Units of 1..16 rows (heads per kv head x new tokens) on both decode
    kernels: ragged stages, empty and one-key sequences, causal token limits,
    each block size."""
    lens = [1, 0, 127, 128, 129, 700, 2049, 3]
    c = fia_inputs.paged_decode_case(len(lens), n1, n2, 128, lens, block_size=bs,
                                     workload=3700 + 10 * n1 + n2 + qs + bs, q_tokens=qs)
    _check_tokens(fia, c, mode)


def test_small_units_full_workload_both_paths(fia, decode_path):
    """The headline paged workload on both kernels: every output."""
    _check_paged(fia, fia_inputs.workload_paged_gqa_decode())


def test_sixteen_row_units_full_workload_both_paths(fia, decode_path):
    """The headline workload with 4 new tokens per sequence (16 rows per
    unit, causal) on both kernels: sampled (batch, head) rows."""
    base = fia_inputs.workload_paged_gqa_decode()
    c = fia_inputs.paged_decode_case(16, 32, 8, 128, base.kv_lens, block_size=128, workload=3400, q_tokens=4)
    rng = np.random.default_rng(11)
    rows = [(int(b), int(h)) for b, h in zip(rng.integers(0, 16, 24), rng.integers(0, 32, 24))]
    rows += [(12, h) for h in range(4)]
    _check_rows(fia, c, rows, mode=3)


def test_small_units_f16_long_split(fia, decode_path):
    """fp16, sequences long enough to be split over many CTAs (merged
    partials), sampled rows."""
    c = fia_inputs.paged_decode_case(8, 32, 8, 128, [16384] * 8, block_size=128, workload=3800, dtype="f16")
    rng = np.random.default_rng(5)
    rows = [(int(b), int(h)) for b, h in zip(rng.integers(0, 8, 24), rng.integers(0, 32, 24))]
    rows += [(0, h) for h in range(4)]
    _check_rows(fia, c, rows)


def test_small_units_timeout_path(fia):
    """The warp-level kernel's waits give up under a 1 ns limit and report
    FIA_ERR_TIMEOUT; the next call is correct."""
    from attention_fia_prefill_gb300 import _binding as B
    lib = B.load_library()
    c = fia_inputs.paged_decode_case(4, 4, 1, 128, [3000, 2000, 4000, 100], workload=3610)
    ws = torch.empty(16 << 20, dtype=torch.uint8, device="cuda")
    lib.fia_debug_set_wait_limit_ns(1)
    try:
        _run_paged(fia, c, workspace=ws)
        status = fia.fia_device_status(ws)
    finally:
        lib.fia_debug_set_wait_limit_ns(0)
    assert status == 10, status
    out, lse = _run_paged(fia, c, workspace=ws)
    assert fia.fia_device_status(ws) == 0
    ro, rl = _oracle_paged(c)
    assert_out_close(out, ro, c.q.dtype)
    assert_lse_close(lse, rl)


# ------------------------------------------------------------ atten_mask (Q_S = 1)
def _mask_for(c, shape_kind, dtype, workload, pad=5, full_batch=1):
    """A random key mask over max(kv_lens) + pad keys in the given form; one
    batch's keys all masked (its rows give 0 and lse +inf)."""
    B, S = len(c.kv_lens), max(c.kv_lens) + pad
    shape = {"b": (B, S), "b1": (B, 1, S), "b11": (B, 1, 1, S), "1": (1, S)}[shape_kind]
    m = fia_inputs.atten_mask(shape, "random", density=0.3, dtype=dtype, workload=workload)
    if full_batch is not None and shape[0] > 1:
        m[full_batch] = True if dtype == "bool" else 1
    return m


def _check_masked(fia, c, mask):
    out, lse = _run_paged(fia, c, atten_mask=mask.cuda())
    ro, rl = fia_oracle.fia_decode(c.q, c.k_pool, c.v_pool, num_heads=c.num_heads,
                                   num_key_value_heads=c.num_key_value_heads, scale_value=c.scale,
                                   input_layout="BNSD", actual_seq_kvlen=c.kv_lens, block_table=c.block_table,
                                   block_size=c.block_size, atten_mask=mask)
    assert_out_close(out, ro, c.q.dtype)
    assert_lse_close(lse, rl)
    return out, lse


# (N1, N2, D, mask form, mask dtype, block size): 4-row and 16-row units on the
# warp-level kernel, 32-row units and head_dim 64 on the tcgen05 kernel
MASK_DECODE_CASES = [(32, 8, 128, "b", "u8", 128), (8, 1, 128, "b1", "bool", 64), (64, 2, 128, "b11", "i8", 16),
                     (8, 2, 64, "1", "u8", 128), (4, 4, 128, "b", "bool", 256)]


@pytest.mark.parametrize("n1,n2,D,form,mdtype,bs", MASK_DECODE_CASES)
def test_decode_atten_mask(fia, n1, n2, D, form, mdtype, bs):
    """atten_mask with one new token: every mask form and dtype, ragged and
    empty sequences, a batch with every key masked, each kernel."""
    lens = [1, 0, 127, 128, 129, 700, 2049, 3]
    c = fia_inputs.paged_decode_case(len(lens), n1, n2, D, lens, block_size=bs, workload=4600 + n1 + D + bs)
    _check_masked(fia, c, _mask_for(c, form, mdtype, 4700 + n1 + bs, full_batch=None if form == "1" else 5))


def test_decode_atten_mask_both_paths_split(fia, decode_path):
    """Long sequences split over many CTAs (merged partials, the tail merge)
    with a key mask, on both kernels; an all-zero mask gives the unmasked
    bits."""
    lens = [16384, 9000, 5000, 1]
    c = fia_inputs.paged_decode_case(len(lens), 32, 8, 128, lens, block_size=128, workload=4800)
    _check_masked(fia, c, _mask_for(c, "b", "u8", 4801, full_batch=3))
    zero = torch.zeros((len(lens), max(lens)), dtype=torch.uint8)
    out_z, lse_z = _run_paged(fia, c, atten_mask=zero.cuda())
    out_n, lse_n = _run_paged(fia, c)
    assert torch.equal(out_z, out_n) and torch.equal(lse_z, lse_n)


"""Prefill parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs, element by element for small cases, on sampled rows at
the full varlen workload."""
import math

import numpy as np
import pytest
import torch

import fia_inputs
from oracle import fia_oracle
from tests.parity import assert_lse_close, assert_out_close, assert_rows_close

pytestmark = pytest.mark.gpu


def _run(fia, case, **kw):
    dev = "cuda"
    q, k, v = case.q.to(dev), case.k.to(dev), case.v.to(dev)
    out, lse = fia.fia_prefill(q, k, v, num_heads=case.num_heads, num_key_value_heads=case.num_key_value_heads,
                               scale_value=case.scale, input_layout=case.layout, sparse_mode=case.sparse_mode,
                               actual_seq_qlen=case.actual_seq_qlen, actual_seq_kvlen=case.actual_seq_kvlen,
                               softmax_lse_flag=True, **kw)
    torch.cuda.synchronize()
    return out, lse


def _oracle(case, rows=None):
    return fia_oracle.fia_prefill(case.q, case.k, case.v, num_heads=case.num_heads,
                                  num_key_value_heads=case.num_key_value_heads, scale_value=case.scale,
                                  input_layout=case.layout, sparse_mode=case.sparse_mode,
                                  actual_seq_qlen=case.actual_seq_qlen, actual_seq_kvlen=case.actual_seq_kvlen,
                                  rows=rows)


def _check_full(fia, case):
    out, lse = _run(fia, case)
    ref_o, ref_l = _oracle(case)
    assert_out_close(out, ref_o, case.q.dtype)
    assert_lse_close(lse, ref_l)
    return out, lse


def test_small_bnsd_f16_causal(fia):
    """Prefill BNSD fp16: B=1, N=2, S=128, D=64, causal, LSE on."""
    _check_full(fia, fia_inputs.workload_prefill_bnsd_f16_small())


@pytest.mark.parametrize("mode", [0, 2, 3])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_gqa_bnsd(fia, mode, D):
    """Several tiles with a ragged tail (S = 300), GQA 4/2, both head dims."""
    case = fia_inputs.prefill_case(2, 4, 2, 300, 300, D, dtype="bf16", layout="BNSD", sparse_mode=mode,
                                   workload=1000 + D + mode)
    _check_full(fia, case)


@pytest.mark.parametrize("mode,D,dtype", [(0, 64, "f16"), (2, 128, "bf16"), (3, 128, "f16")])
def test_long_rows_ring_reuse(fia, mode, D, dtype):
    """1000 query rows x 1100 keys: query-tile pairs with a ragged last pair,
    nine K/V tiles cycling through the shared-memory ring several times."""
    case = fia_inputs.prefill_case(1, 2, 1, 1000, 1100, D, dtype=dtype, layout="BNSD", sparse_mode=mode,
                                   workload=1700 + D + mode)
    _check_full(fia, case)


def test_pfa_example_shape_f16(fia):
    """npu_prompt_flash_attention call example: q (1,8,164,128) vs k/v (1,8,1024,128), fp16."""
    case = fia_inputs.prefill_case(1, 8, 8, 164, 1024, 128, dtype="f16", layout="BNSD", workload=7)
    out, _ = _check_full(fia, case)
    assert out.shape == (1, 8, 164, 128) and out.dtype == torch.float16


@pytest.mark.parametrize("sq,skv", [(100, 300), (300, 100), (1, 257)])
def test_right_down_causal_unequal(fia, sq, skv):
    """sparse_mode 3 aligns the diagonal to the bottom-right corner; with
    S_q > S_kv the leading rows have no key (0 / +inf)."""
    case = fia_inputs.prefill_case(1, 2, 1, sq, skv, 128, dtype="bf16", layout="BNSD", sparse_mode=3,
                                   workload=1100 + sq)
    _check_full(fia, case)


@pytest.mark.parametrize("layout", ["BSND", "BSH"])
def test_layouts(fia, layout):
    case = fia_inputs.prefill_case(2, 4, 1, 190, 190, 128, dtype="f16", layout=layout, sparse_mode=2,
                                   workload=1200)
    _check_full(fia, case)


def test_actual_lengths_with_poisoned_padding(fia):
    """actual_seq lengths shorter than S; K/V padding rows are NaN and must not
    reach the output; query padding rows come back as 0 / +inf."""
    case = fia_inputs.prefill_case(3, 2, 2, 260, 260, 128, dtype="bf16", layout="BNSD", sparse_mode=0,
                                   actual_seq_qlen=[260, 5, 130], actual_seq_kvlen=[200, 1, 259],
                                   poison_padding=True, workload=1300)
    _check_full(fia, case)


def test_tnd_varlen_small(fia):
    """TND with lengths around tile boundaries, including an empty sequence."""
    lens = [1, 127, 128, 0, 129, 300]
    case = fia_inputs.tnd_case(lens, lens, 8, 2, 128, "bf16", sparse_mode=3, workload=1400)
    _check_full(fia, case)


def test_tnd_dense_unequal_lists(fia):
    case = fia_inputs.tnd_case([50, 200], [300, 70], 4, 4, 64, "f16", sparse_mode=0, workload=1401)
    _check_full(fia, case)


def test_empty_kv(fia):
    """K/V with S2 = 0: out all zeros, lse all +inf (the pages' empty rule)."""
    q = torch.randn(1, 2, 5, 64, dtype=torch.float16, device="cuda")
    k = torch.zeros(1, 2, 0, 64, dtype=torch.float16, device="cuda")
    out, lse = fia.fia_prefill(q, k, k, num_heads=2, input_layout="BNSD", softmax_lse_flag=True, scale_value=0.125)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(torch.isinf(lse) & (lse > 0))


def test_empty_query_is_noop(fia):
    q = torch.zeros(0, 2, 5, 64, dtype=torch.float16, device="cuda")
    out, _ = fia.fia_prefill(q, q, q, num_heads=2, input_layout="BNSD")
    assert out.numel() == 0


def test_deterministic(fia):
    """Repeated calls are bitwise identical (the pages' operator is deterministic)."""
    case = fia_inputs.tnd_case([333, 700], [333, 700], 8, 2, 128, "bf16", sparse_mode=3, workload=1500)
    o1, l1 = _run(fia, case)
    o2, l2 = _run(fia, case)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gqa_equals_repeated_heads(fia):
    case = fia_inputs.prefill_case(1, 8, 2, 257, 257, 128, dtype="bf16", layout="BNSD", sparse_mode=2,
                                   workload=1600)
    o1, l1 = _run(fia, case)
    rep = fia_inputs.PrefillCase(case.q, case.k.repeat_interleave(4, dim=1), case.v.repeat_interleave(4, dim=1),
                                 8, 8, case.scale, "BNSD", 2)
    o2, l2 = _run(fia, rep)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_full_tnd_varlen_workload_sampled(fia):
    """Varlen TND bf16: 8 sequences with lengths uniform on [256, 4096], GQA
    32/8, D=128, causal, LSE on -- at full size, one row of every work item
    (2272 rows) vs the oracle."""
    case = fia_inputs.workload_tnd_varlen()
    out, lse = _run(fia, case)
    lens = [b - a for a, b in zip([0] + case.actual_seq_qlen[:-1], case.actual_seq_qlen)]
    starts = [0] + case.actual_seq_qlen[:-1]
    rng = np.random.default_rng(0)
    # one row of every work item (256 query rows of one head), its position
    # cycling over the two tiles' first and last rows and a random one
    rows = []
    for b in range(len(lens)):
        for q0 in range(0, lens[b], 256):
            for h in range(32):
                pick = (q0, q0 + 127, q0 + 128, q0 + 255, q0 + int(rng.integers(256)))[(h + q0 // 256) % 5]
                rows.append((b, h, min(pick, lens[b] - 1)))
    ref = _oracle(case, rows=rows)
    assert_rows_close(out, lse, rows, ref, lambda r: (starts[r[0]] + r[2], r[1]), torch.bfloat16)
    assert torch.isfinite(out.float()).all()


# ------------------------------------------------------------- band (mode 4)
def _check_band(fia, case, pre, nxt):
    out, lse = _run(fia, case, pre_tokens=pre, next_tokens=nxt)
    ref_o, ref_l = fia_oracle.fia_prefill(case.q, case.k, case.v, num_heads=case.num_heads,
                                          num_key_value_heads=case.num_key_value_heads, scale_value=case.scale,
                                          input_layout=case.layout, sparse_mode=4,
                                          actual_seq_qlen=case.actual_seq_qlen,
                                          actual_seq_kvlen=case.actual_seq_kvlen, pre_tokens=pre, next_tokens=nxt)
    assert_out_close(out, ref_o, case.q.dtype)
    assert_lse_close(lse, ref_l)


@pytest.mark.parametrize("sq,skv,pre,nxt,D", [(300, 300, 100, 50, 128), (200, 500, 64, 0, 128), (700, 600, 130, 260, 64),
                                              (520, 520, 0, 0, 128), (300, 300, 2000, 2000, 64)])
def test_band(fia, sq, skv, pre, nxt, D):
    """sparse_mode 4: row i sees keys i + S_kv - S_q - pre .. i + S_kv - S_q + next
    (both edges inside a tile, a band narrower than a tile, a band wider than
    the sequence)."""
    case = fia_inputs.prefill_case(2, 4, 2, sq, skv, D, dtype="bf16", layout="BNSD", sparse_mode=4,
                                   workload=1800 + sq + pre)
    _check_band(fia, case, pre, nxt)


def test_band_tnd_varlen(fia):
    lens = [1, 127, 300, 0, 1000, 129]
    case = fia_inputs.tnd_case(lens, lens, 8, 2, 128, "bf16", sparse_mode=4, workload=1900)
    _check_band(fia, case, 256, 32)


# ------------------------------------------------------------ explicit atten_mask
def _check_mask(fia, case, mask, pre=2147483647, nxt=2147483647):
    out, lse = _run(fia, case, atten_mask=mask.to("cuda"), pre_tokens=pre, next_tokens=nxt)
    ref_o, ref_l = fia_oracle.fia_prefill(case.q, case.k, case.v, num_heads=case.num_heads,
                                          num_key_value_heads=case.num_key_value_heads, scale_value=case.scale,
                                          input_layout=case.layout, sparse_mode=case.sparse_mode, atten_mask=mask,
                                          actual_seq_qlen=case.actual_seq_qlen,
                                          actual_seq_kvlen=case.actual_seq_kvlen, pre_tokens=pre, next_tokens=nxt)
    assert_out_close(out, ref_o, case.q.dtype)
    assert_lse_close(lse, ref_l)
    return out, lse


# (mode, D, dtype, mask shape (B=2, S1=300, S2=260 + pad), mask dtype, kind, pre, next).  The
# padding of the key axis picks the copy granule: 260 -> 4 bytes, 264 -> 8, 272 -> 16, 261 -> 1.
MASK_CASES = [
    (1, 128, "bf16", (300, 272), "u8", "random", None, None),
    (1, 64, "f16", (2, 300, 264), "bool", "blocks", None, None),
    (1, 128, "bf16", (1, 300, 260), "i8", "blocks", None, None),
    (0, 128, "bf16", (2, 1, 300, 261), "u8", "random", 100, 20),
    (0, 64, "bf16", (1, 1, 304, 272), "bool", "blocks", None, None),
    (0, 128, "f16", (300, 264), "i8", "random", 0, 300),
]


@pytest.mark.parametrize("mode,D,dtype,mshape,mdtype,kind,pre,nxt", MASK_CASES)
def test_explicit_mask(fia, mode, D, dtype, mshape, mdtype, kind, pre, nxt):
    """sparse_mode 1 (mask alone) and 0 (mask and the pre/next window): every
    mask shape the pages list, bool / int8 / uint8 with assorted nonzero bytes,
    each copy granule, ragged query and key tails, fully masked rows."""
    case = fia_inputs.prefill_case(2, 4, 2, 300, 260, D, dtype=dtype, layout="BNSD", sparse_mode=mode,
                                   workload=2000 + D + mode + mshape[-1])
    mask = fia_inputs.atten_mask(mshape, kind, dtype=mdtype, workload=2100 + mshape[-1])
    kw = {} if pre is None else {"pre": pre, "nxt": nxt}
    _check_mask(fia, case, mask, **kw)


def test_mask_causal_equals_mode2(fia):
    """A lower-triangular mask in sparse_mode 1 gives the same bits as sparse_mode 2
    (tiles past the diagonal only add exact zeros), and an all-zero mask in
    sparse_mode 0 the same bits as no mask."""
    case = fia_inputs.prefill_case(1, 4, 2, 700, 700, 128, dtype="bf16", layout="BNSD", sparse_mode=1, workload=2200)
    causal = fia_inputs.atten_mask((700, 704), "causal")
    out_m, lse_m = _run(fia, case, atten_mask=causal.cuda())
    case.sparse_mode = 2
    out_c, lse_c = _run(fia, case)
    assert torch.equal(out_m, out_c) and torch.equal(lse_m, lse_c)
    case.sparse_mode = 0
    out_z, lse_z = _run(fia, case, atten_mask=torch.zeros((700, 700), dtype=torch.bool, device="cuda"))
    out_d, lse_d = _run(fia, case)
    assert torch.equal(out_z, out_d) and torch.equal(lse_z, lse_d)


def test_mask_tnd_varlen(fia):
    """TND: the mask is indexed with each sequence's own row / key numbers."""
    lens_q, lens_kv = [1, 127, 300, 0, 700, 129], [5, 127, 260, 3, 700, 200]
    case = fia_inputs.tnd_case(lens_q, lens_kv, 8, 2, 128, "bf16", sparse_mode=1, workload=2300)
    mask = fia_inputs.atten_mask((6, 700, 704), "blocks", workload=2301)
    _check_mask(fia, case, mask)


def test_mask_2k_full(fia):
    """2048 x 2048 with a tile-structured mask (visible, masked and random
    tiles): sixteen K/V tiles through the ring, element by element."""
    case = fia_inputs.prefill_case(1, 8, 2, 2048, 2048, 128, dtype="bf16", layout="BNSD", sparse_mode=1, workload=2400)
    mask = fia_inputs.atten_mask((2048, 2048), "blocks", workload=2401)
    _check_mask(fia, case, mask)


def test_mask_tile_codes_shape_the_walk(fia):
    """Tile codes of the mask decide each pair's walk: a query tile with every
    key masked (tile A of the first pair: no keys at all), a walk that starts
    late (tile B's first visible tile is the fourth), fully masked tiles inside
    a walk (P = 0 there), a tile B with every key masked (it still walks tile
    A's range), and mixed tiles; fully masked rows give 0 and lse = +inf."""
    S, T = 640, 128
    case = fia_inputs.prefill_case(1, 4, 2, S, S, 128, dtype="bf16", layout="BNSD", sparse_mode=1, workload=2450)
    g = np.random.default_rng(2451)
    visible = {(1, 3): "all", (2, 1): "all", (2, 4): "mixed", (4, 0): "mixed", (4, 2): "all"}
    m = np.ones((S, S), dtype=np.uint8)
    for (qt, kt), kind in visible.items():
        blk = np.zeros((T, T), dtype=np.uint8) if kind == "all" else (g.random((T, T)) < 0.5).astype(np.uint8)
        m[qt * T:(qt + 1) * T, kt * T:(kt + 1) * T] = blk
    _check_mask(fia, case, torch.from_numpy(m))


def test_full_tnd_band_and_mask_workloads_sampled(fia):
    """The varlen TND workload at full size with the band of the bench
    (sparse_mode 4, pre_tokens 1024, next_tokens 0) and with an explicit
    uint8 causal mask (sparse_mode 1, a (4096, 4096) mask): sampled rows
    against the oracle."""
    case = fia_inputs.workload_tnd_varlen()
    lens = [b - a for a, b in zip([0] + case.actual_seq_qlen[:-1], case.actual_seq_qlen)]
    starts = [0] + case.actual_seq_qlen[:-1]
    rng = np.random.default_rng(7)
    rows = []
    for b in range(len(lens)):
        for i in sorted({0, lens[b] - 1, int(rng.integers(lens[b])), 1024, 1100}):
            if i < lens[b]:
                rows.append((b, int(rng.integers(32)), i))
    index = lambda r: (starts[r[0]] + r[2], r[1])
    kw_oracle = dict(num_heads=case.num_heads, num_key_value_heads=case.num_key_value_heads, scale_value=case.scale,
                     input_layout="TND", actual_seq_qlen=case.actual_seq_qlen, actual_seq_kvlen=case.actual_seq_kvlen,
                     rows=rows)
    case.sparse_mode = 4
    out, lse = _run(fia, case, pre_tokens=1024, next_tokens=0)
    ref = fia_oracle.fia_prefill(case.q, case.k, case.v, sparse_mode=4, pre_tokens=1024, next_tokens=0, **kw_oracle)
    assert_rows_close(out, lse, rows, ref, index, torch.bfloat16)
    mask = fia_inputs.atten_mask((4096, 4096), "causal")
    case.sparse_mode = 1
    out, lse = _run(fia, case, atten_mask=mask.cuda())
    ref = fia_oracle.fia_prefill(case.q, case.k, case.v, sparse_mode=1, atten_mask=mask, **kw_oracle)
    assert_rows_close(out, lse, rows, ref, index, torch.bfloat16)

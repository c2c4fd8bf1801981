"""The C-ABI library on the host, without a GPU: it loads, exports every symbol
include/fia.h declares, and rejects invalid arguments with the documented
status codes before any CUDA call (validation rules from the pages: GQA head
rules, actual_seq list rules, TND cumulative lists, rope pairing, sparse_mode
range, block_table shape, block-sparse constraints)."""
import ctypes
import os
import re
import subprocess

import pytest

from attention_fia_prefill_gb300 import _binding as B
from attention_fia_prefill_gb300 import build as fia_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
P = 1 << 20          # a fake, 16-byte aligned device address (never dereferenced)


@pytest.fixture(scope="module")
def lib():
    fia_build.build()
    return B.load_library()


def header_symbols():
    src = open(os.path.join(ROOT, "include", "fia.h")).read()
    return re.findall(r"FIA_API\s+[\w\s\*]+?\b(\w+)\s*\(", src)


def test_exports_every_declared_symbol(lib):
    declared = header_symbols()
    assert set(declared) == set(B.EXPORTS)
    out = subprocess.run(["nm", "-D", "--defined-only", fia_build.LIB], capture_output=True, text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared:
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_status_strings(lib):
    for code, name in B.STATUS_NAMES.items():
        assert lib.fia_status_string(code).decode().startswith(name)


def t(shape, dtype=B.DTYPE_BF16, ptr=P):
    return B.raw_desc(ptr, dtype, shape)


def params(lib, **kw):
    return B.Params(**kw)


def prefill_ws(lib, q, k, v, prm, out=None, lse=None, mask=None):
    ws = ctypes.c_size_t(0)
    r = lib.fia_prefill_get_workspace_size(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v),
                                           ctypes.byref(mask) if mask else None, ctypes.byref(prm.p),
                                           ctypes.byref(out or q), ctypes.byref(lse) if lse else None,
                                           ctypes.byref(ws))
    return r, ws.value


def test_prefill_valid_reports_workspace(lib):
    q, k = t((2, 4, 300, 128)), t((2, 2, 300, 128))
    r, ws = prefill_ws(lib, q, k, k, params(lib, num_heads=4, num_key_value_heads=2, input_layout="BNSD",
                                            sparse_mode=3, scale_value=0.08))
    assert r == B.FIA_OK and ws >= 256 + 2 * 3 * 4 * 16


def test_empty_query_ok(lib):
    q = t((0, 4, 5, 128))
    r, ws = prefill_ws(lib, q, q, q, params(lib, num_heads=4, input_layout="BNSD"))
    assert r == B.FIA_OK and ws == 256


@pytest.mark.parametrize("n1,n2,code", [(6, 4, 11), (130, 2, 11), (4, 0, 0), (0, 1, 11)])
def test_gqa_head_rules(lib, n1, n2, code):
    """Q_N must be a multiple of KV_N with ratio <= 64; KV_N = 0 means Q_N."""
    kvn = n2 if n2 else n1
    q, k = t((1, max(n1, 1), 8, 128)), t((1, max(kvn, 1), 8, 128))
    r, _ = prefill_ws(lib, q, k, k, params(lib, num_heads=n1, num_key_value_heads=n2, input_layout="BNSD"))
    assert r == code


@pytest.mark.parametrize("qlen,code", [([3], 0), ([3, 4, 5], 0), ([3, 4], 6), ([9], 6), ([-1], 6)])
def test_actual_seq_list_rules(lib, qlen, code):
    """A list of 1 is broadcast; >= B takes the first B; other counts and
    entries outside [0, S] are errors."""
    q = t((3, 2, 8, 64))
    r, _ = prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="BNSD", actual_seq_qlen=qlen))
    assert r == code


def test_tnd_lists(lib):
    q = t((10, 2, 64))
    r, _ = prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="TND"))
    assert r == B.FIA_ERR_SEQLEN if hasattr(B, "FIA_ERR_SEQLEN") else r == 6
    r, _ = prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="TND", actual_seq_qlen=[4, 3],
                                           actual_seq_kvlen=[4, 10]))
    assert r == 6
    r, _ = prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="TND", actual_seq_qlen=[4, 11],
                                           actual_seq_kvlen=[4, 10]))
    assert r == 6
    r, ws = prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="TND", actual_seq_qlen=[4, 10],
                                            actual_seq_kvlen=[4, 10], sparse_mode=3))
    assert r == 0 and ws > 256


@pytest.mark.parametrize("mode,code", [(9, 12), (5, 12), (-1, 12), (4, 0), (1, 12), (0, 0), (2, 0), (3, 0)])
def test_sparse_mode_range(lib, mode, code):
    q = t((1, 2, 8, 64))
    r, _ = prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="BNSD", sparse_mode=mode))
    assert r == code


def test_causal_mask_shape(lib):
    """Modes 2/3 accept no mask, or the (2048, 2048) form; other shapes are errors."""
    q = t((1, 2, 8, 64))
    m_ok, m_bad = t((2048, 2048), B.DTYPE_BOOL), t((8, 8), B.DTYPE_BOOL)
    assert prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="BNSD", sparse_mode=2), mask=m_ok)[0] == 0
    assert prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="BNSD", sparse_mode=2), mask=m_bad)[0] == 12


def test_explicit_mask_rules(lib):
    """Modes 0 / 1 with an explicit atten_mask: bool / int8 / uint8 in the shapes
    (S1,S2), (B|1,S1,S2), (B|1,1,S1,S2) covering the query / key lengths."""
    q, k = t((2, 2, 8, 64)), t((2, 2, 10, 64))

    def ws(mode, mask):
        return prefill_ws(lib, q, k, k, params(lib, num_heads=2, input_layout="BNSD", sparse_mode=mode), mask=mask)[0]

    for dt in (B.DTYPE_BOOL, B.DTYPE_U8, B.DTYPE_I8):
        for shape in ((8, 10), (2, 8, 10), (1, 8, 10), (2, 1, 8, 10), (1, 1, 8, 16), (9, 11)):
            assert ws(1, t(shape, dt)) == 0 and ws(0, t(shape, dt)) == 0, (dt, shape)
    assert ws(1, t((8, 10), B.DTYPE_F16)) == 2        # element type
    assert ws(1, t((7, 10), B.DTYPE_U8)) == 3         # fewer rows than S1
    assert ws(1, t((8, 9), B.DTYPE_U8)) == 3          # fewer columns than S2
    assert ws(1, t((3, 8, 10), B.DTYPE_U8)) == 3      # batch dim neither 1 nor B
    assert ws(1, t((2, 2, 8, 10), B.DTYPE_U8)) == 3   # head dim must be 1
    assert ws(1, t((10,), B.DTYPE_U8)) == 3           # rank
    assert ws(1, None) == 12                          # mode 1 needs the mask


def test_paged_prefill_rules(lib):
    """Prefill against a paged cache: block_size 128..512 in steps of 128,
    actual_seq_kvlen required, block_table (B, >= max blocks) int32, blocknum
    covering the lengths, one table row per TND sequence."""
    q = t((2, 4, 300, 128))
    kp = t((9, 2, 256, 128))

    def ws(q, kp, table, bs=256, kv=(500, 300), layout="BNSD", ql=None):
        prm = params(lib, num_heads=4, num_key_value_heads=2, input_layout=layout, sparse_mode=3, block_size=bs,
                     actual_seq_kvlen=list(kv) if kv is not None else None, actual_seq_qlen=ql)
        w = ctypes.c_size_t(0)
        return lib.fia_prefill_paged_get_workspace_size(ctypes.byref(q), ctypes.byref(kp), ctypes.byref(kp),
                                                        ctypes.byref(table), None, ctypes.byref(prm.p),
                                                        ctypes.byref(q), None, ctypes.byref(w))

    tab = t((2, 3), B.DTYPE_I32)
    assert ws(q, kp, tab) == 0
    assert ws(q, t((9, 256, 256)), tab) == 0                      # (blocknum, bs, KV_N*D)
    assert ws(q, t((9, 2, 128, 128)), tab, bs=128) == 6             # 500 keys > 3 table columns x 128
    assert ws(q, t((9, 2, 64, 128)), tab, bs=64) == 7               # block_size below 128
    assert ws(q, t((9, 2, 640, 128)), tab, bs=640) == 7             # above 512
    assert ws(q, t((3, 2, 256, 128)), tab) == 7                     # 3 blocks < 2 + 2 needed
    assert ws(q, kp, t((2, 3), B.DTYPE_I64)) == 7                   # table dtype
    assert ws(q, kp, t((3, 3), B.DTYPE_I32)) == 3                   # table rows != B
    assert ws(q, kp, tab, kv=None) == 6                             # actual_seq_kvlen required
    assert ws(q, t((9, 2, 256, 128)), tab, bs=128) == 3             # pool block dim != block_size
    qt = t((800, 4, 128))
    assert ws(qt, kp, tab, layout="TND", ql=[300, 800]) == 0
    assert ws(qt, kp, t((3, 3), B.DTYPE_I32), layout="TND", ql=[300, 800]) == 7


def test_mla_prefill_rules(lib):
    """MLA prefill: query/key D 192 without rope tensors, or D 128 with both
    (D 64); value and output D 128; an explicit mask is taken as for the
    plain prefill (a mask too short for the keys is refused)."""
    def ws(q, k, v, out, qr=None, kr=None, mask=None, mode=3):
        prm = params(lib, num_heads=4, num_key_value_heads=2, input_layout="TND", sparse_mode=mode,
                     actual_seq_qlen=[100, 300], actual_seq_kvlen=[100, 300])
        w = ctypes.c_size_t(0)
        ref = lambda d: ctypes.byref(d) if d is not None else None
        return lib.fia_prefill_mla_get_workspace_size(ref(q), ref(k), ref(v), ref(qr), ref(kr), ref(mask),
                                                      ctypes.byref(prm.p), ref(out), None, ctypes.byref(w))

    q192, k192, v, out = t((300, 4, 192)), t((300, 2, 192)), t((300, 2, 128)), t((300, 4, 128))
    q128, k128, qr, kr = t((300, 4, 128)), t((300, 2, 128)), t((300, 4, 64)), t((300, 2, 64))
    assert ws(q192, k192, v, out) == 0
    assert ws(q128, k128, v, out, qr, kr) == 0
    assert ws(q128, k128, v, out) == 5                           # D 128 needs the rope tensors
    assert ws(q192, k192, v, out, qr, kr) == 5                   # D 192 takes none
    assert ws(q128, k128, v, out, qr, None) == 3                 # both or neither
    assert ws(q192, k192, t((300, 2, 192)), out) == 5            # value D 128 only
    assert ws(q192, k192, v, t((300, 4, 192))) == 3              # output has value's D
    assert ws(q128, k128, v, out, t((300, 4, 32)), kr) == 3      # rope D 64
    assert ws(q192, k192, v, out, mask=t((300, 300), B.DTYPE_U8), mode=1) == 0
    assert ws(q128, k128, v, out, qr, kr, mask=t((2, 1, 300, 300), B.DTYPE_BOOL), mode=0) == 0
    assert ws(q192, k192, v, out, mask=t((300, 150), B.DTYPE_U8), mode=1) != 0   # keys up to 200


def test_bsa_fp8_rules(lib):
    """FP8 block-sparse: e4m3 query/key/value, D 128, bf16 output, block shape
    [128, 256 | 512], fp32 scales (B, N1, ceil(S1/128), 1) / (B, N2, ceil(S2/Y), 1)."""
    F8, F32 = B.DTYPE_F8E4M3, B.DTYPE_F32
    q, k = t((2, 4, 300, 128), F8), t((2, 2, 600, 128), F8)
    out = t((2, 4, 300, 128), B.DTYPE_BF16)
    mask = t((2, 4, 3, 3), B.DTYPE_U8)
    qs, ks = t((2, 4, 3, 1), F32), t((2, 2, 3, 1), F32)

    def ws(q=q, k=k, out=out, mask=mask, shape=(128, 256), qs=qs, ks=ks, vs=ks):
        prm = params(lib, num_heads=4, num_key_value_heads=2, input_layout="BNSD")
        w = ctypes.c_size_t(0)
        bs = (ctypes.c_int64 * 2)(*shape)
        ref = lambda d: ctypes.byref(d) if d is not None else None
        return lib.bsa_fp8_get_workspace_size(ref(q), ref(k), ref(k), ref(mask), bs, ref(qs), ref(ks), ref(vs),
                                              ctypes.byref(prm.p), ref(out), None, ctypes.byref(w))

    assert ws() == 0
    assert ws(mask=t((2, 4, 3, 2), B.DTYPE_U8), shape=(128, 512), ks=t((2, 2, 2, 1), F32),
              vs=t((2, 2, 2, 1), F32)) == 0
    assert ws(out=t((2, 4, 300, 128), B.DTYPE_F16)) == 2        # output bf16
    assert ws(q=t((2, 4, 300, 128), B.DTYPE_BF16)) == 2         # all three e4m3
    assert ws(shape=(128, 128), mask=t((2, 4, 3, 5), B.DTYPE_U8)) == 3   # Y 256 / 512 only
    assert ws(qs=t((2, 4, 2, 1), F32)) == 3                     # query blocks of 128 rows
    assert ws(ks=t((2, 2, 3, 1), B.DTYPE_F16)) == 3             # fp32 scales
    assert ws(vs=None) == 1                                     # all three scales
    q64, k64 = t((2, 4, 300, 64), F8), t((2, 2, 600, 64), F8)
    assert ws(q=q64, k=k64, out=t((2, 4, 300, 64), B.DTYPE_BF16)) == 5   # D 128 only
    assert ws(mask=None) == 0                                   # no mask: dense FP8 attention


def test_paged_prefill_with_mask_and_tnd_fp8_scales(lib):
    """Paged prefill takes an explicit mask covering the per-batch lengths;
    FP8 block-sparse in TND sizes its scale blocks by the longest sequence."""
    q, kp, tab = t((2, 4, 300, 128)), t((9, 2, 256, 128)), t((2, 3), B.DTYPE_I32)

    def ws_paged(mask, mode=1):
        prm = params(lib, num_heads=4, num_key_value_heads=2, input_layout="BNSD", sparse_mode=mode, block_size=256,
                     actual_seq_kvlen=[500, 300])
        w = ctypes.c_size_t(0)
        return lib.fia_prefill_paged_get_workspace_size(ctypes.byref(q), ctypes.byref(kp), ctypes.byref(kp),
                                                        ctypes.byref(tab), ctypes.byref(mask) if mask else None,
                                                        ctypes.byref(prm.p), ctypes.byref(q), None,
                                                        ctypes.byref(w))

    assert ws_paged(t((300, 512), B.DTYPE_U8)) == 0
    assert ws_paged(t((300, 499), B.DTYPE_U8)) == 3       # shorter than the 500 keys of batch 0
    assert ws_paged(None) == 12                           # mode 1 needs a mask

    F8, F32 = B.DTYPE_F8E4M3, B.DTYPE_F32
    # TND: sequences of 100 and 700 rows, so 6 query blocks and 3 key blocks at the longest
    qt, kt = t((800, 4, 128), F8), t((800, 2, 128), F8)
    out = t((800, 4, 128), B.DTYPE_BF16)
    mask = t((2, 4, 6, 3), B.DTYPE_U8)                    # ceil(700/128) x ceil(700/256)

    def ws_fp8(qs, ks):
        prm = params(lib, num_heads=4, num_key_value_heads=2, input_layout="TND", actual_seq_qlen=[100, 800],
                     actual_seq_kvlen=[100, 800])
        w = ctypes.c_size_t(0)
        bs = (ctypes.c_int64 * 2)(128, 256)
        return lib.bsa_fp8_get_workspace_size(ctypes.byref(qt), ctypes.byref(kt), ctypes.byref(kt),
                                              ctypes.byref(mask), bs, ctypes.byref(qs), ctypes.byref(ks),
                                              ctypes.byref(ks), ctypes.byref(prm.p), ctypes.byref(out), None,
                                              ctypes.byref(w))

    assert ws_fp8(t((2, 4, 6, 1), F32), t((2, 2, 3, 1), F32)) == 0
    assert ws_fp8(t((2, 4, 7, 1), F32), t((2, 2, 3, 1), F32)) == 3


def test_mla_prefill_modes_and_masks(lib):
    """MLA prefill runs on contiguous key/value only (its entry takes no block
    table); causal and band modes and an explicit mask (modes 0 and 1) are
    taken."""
    q, k, v, out = t((300, 4, 192)), t((300, 2, 192)), t((300, 2, 128)), t((300, 4, 128))

    def ws(mode, mask=None, **kw):
        prm = params(lib, num_heads=4, num_key_value_heads=2, input_layout="TND", sparse_mode=mode,
                     actual_seq_qlen=[300], actual_seq_kvlen=[300], **kw)
        w = ctypes.c_size_t(0)
        return lib.fia_prefill_mla_get_workspace_size(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), None, None,
                                                      ctypes.byref(mask) if mask else None, ctypes.byref(prm.p),
                                                      ctypes.byref(out), None, ctypes.byref(w))

    assert ws(2) == 0 and ws(3) == 0 and ws(4, pre_tokens=64, next_tokens=0) == 0
    assert ws(0, t((300, 300), B.DTYPE_BOOL)) == 0 and ws(1, t((1, 300, 300), B.DTYPE_U8)) == 0
    assert ws(1) != 0   # sparse_mode 1 needs the mask


def test_shape_dtype_layout_errors(lib):
    q, k = t((1, 2, 8, 64)), t((1, 2, 9, 64))
    assert prefill_ws(lib, q, k, q, params(lib, num_heads=2, input_layout="BNSD"))[0] == 3      # k != v
    kf = t((1, 2, 8, 64), B.DTYPE_F16)
    assert prefill_ws(lib, q, kf, kf, params(lib, num_heads=2, input_layout="BNSD"))[0] == 2    # dtype
    assert prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="XYZ"))[0] == 4        # layout
    q96 = t((1, 2, 8, 96))
    assert prefill_ws(lib, q96, q96, q96, params(lib, num_heads=2, input_layout="BNSD"))[0] == 5  # head dim
    qa = t((1, 2, 8, 64), ptr=P + 8)
    assert prefill_ws(lib, qa, qa, qa, params(lib, num_heads=2, input_layout="BNSD"))[0] == 13   # alignment
    lse_bad = t((1, 2, 8), B.DTYPE_F32)
    assert prefill_ws(lib, q, q, q, params(lib, num_heads=2, input_layout="BNSD", softmax_lse_flag=True),
                      lse=lse_bad)[0] == 3


def test_workspace_too_small_rejected_before_launch(lib):
    q = t((1, 2, 8, 64))
    prm = params(lib, num_heads=2, input_layout="BNSD")
    r = lib.fia_prefill(ctypes.byref(q), ctypes.byref(q), ctypes.byref(q), None, ctypes.byref(prm.p),
                        ctypes.byref(q), None, ctypes.c_void_p(P), ctypes.c_size_t(16), None)
    assert r == 8


def decode_ws(lib, q, k, v, prm, qr=None, kr=None, table=None, out=None, mask=None):
    ws = ctypes.c_size_t(0)
    ref = lambda d: ctypes.byref(d) if d is not None else None
    r = lib.fia_decode_get_workspace_size(ref(q), ref(k), ref(v), ref(qr), ref(kr), ref(table), ref(mask),
                                          ctypes.byref(prm.p), ref(out or q), None, ctypes.byref(ws))
    return r, ws.value


def test_decode_mask_rules(lib):
    """Decode atten_mask (Q_S = 1): (B, KV_S), (B, 1, KV_S), (B, 1, 1, KV_S),
    batch dim B or 1, bool / int8 / uint8, at least the longest sequence's
    keys; Q_S > 1 or MLA with a mask are not implemented."""
    q = t((4, 8, 1, 128))
    pool = t((40, 2, 128, 128))
    table = t((4, 10), B.DTYPE_I32)
    ok = params(lib, num_heads=8, num_key_value_heads=2, input_layout="BNSD", block_size=128,
                actual_seq_kvlen=[100, 1000, 1, 1280])
    w = lambda m, qq=q, prm=ok: decode_ws(lib, qq, pool, pool, prm, table=table, mask=m)[0]
    assert w(t((4, 1280), B.DTYPE_U8)) == 0
    assert w(t((4, 1, 1300), B.DTYPE_BOOL)) == 0
    assert w(t((1, 1, 1, 1280), B.DTYPE_I8)) == 0
    assert w(t((4, 1279), B.DTYPE_U8)) == 3                       # shorter than the longest sequence
    assert w(t((3, 1280), B.DTYPE_U8)) == 3                       # batch dim neither B nor 1
    assert w(t((4, 2, 1280), B.DTYPE_U8)) == 3                    # middle dims must be 1
    assert w(t((4, 1, 1, 1, 1280), B.DTYPE_U8)) == 3              # at most 4-D
    assert w(t((4, 1280), B.DTYPE_F16)) == 2                      # dtype
    q3 = t((4, 8, 3, 128))
    prm3 = params(lib, num_heads=8, num_key_value_heads=2, input_layout="BNSD", block_size=128, sparse_mode=3,
                  actual_seq_kvlen=[100, 1000, 1, 1280])
    assert w(t((4, 1280), B.DTYPE_U8), q3, prm3) == 5              # Q_S > 1
    qm = t((2, 1, 128, 512))
    lat = t((16, 128, 512))
    prm = params(lib, num_heads=128, num_key_value_heads=1, input_layout="BSND", block_size=128,
                 actual_seq_kvlen=[256])
    r, _ = decode_ws(lib, qm, lat, lat, prm, qr=t((2, 1, 128, 64)), kr=t((16, 128, 64)),
                     table=t((2, 2), B.DTYPE_I32), mask=t((2, 256), B.DTYPE_U8))
    assert r == 5                                                  # MLA


def test_decode_paged_rules(lib):
    q = t((4, 8, 1, 128))
    pool = t((40, 2, 128, 128))
    table = t((4, 10), B.DTYPE_I32)
    ok = params(lib, num_heads=8, num_key_value_heads=2, input_layout="BNSD", block_size=128,
                actual_seq_kvlen=[100, 1000, 1, 1280])
    r, ws = decode_ws(lib, q, pool, pool, ok, table=table)
    assert r == 0 and ws > 256
    # block_table without actual_seq_kvlen
    r, _ = decode_ws(lib, q, pool, pool, params(lib, num_heads=8, num_key_value_heads=2, input_layout="BNSD",
                                                block_size=128), table=table)
    assert r == 6
    # block_table must be 2-D with first dim B
    assert decode_ws(lib, q, pool, pool, ok, table=t((4, 10, 1), B.DTYPE_I32))[0] == 7
    assert decode_ws(lib, q, pool, pool, ok, table=t((3, 10), B.DTYPE_I32))[0] == 7
    # second dim below maxBlocksPerSeq (1280 tokens need 10 blocks)
    assert decode_ws(lib, q, pool, pool, ok, table=t((4, 9), B.DTYPE_I32))[0] in (6, 7)
    # block_size must fit the cache and be 16-aligned
    bad = params(lib, num_heads=8, num_key_value_heads=2, input_layout="BNSD", block_size=100,
                 actual_seq_kvlen=[100, 1000, 1, 1280])
    assert decode_ws(lib, q, pool, pool, bad, table=table)[0] == 7


def test_decode_rope_pairing(lib):
    q = t((2, 1, 128, 512))
    lat = t((16, 128, 512))
    prm = params(lib, num_heads=128, num_key_value_heads=1, input_layout="BSND", block_size=128,
                 actual_seq_kvlen=[256])
    r, _ = decode_ws(lib, q, lat, lat, prm, qr=t((2, 1, 128, 64)), kr=None, table=t((2, 2), B.DTYPE_I32))
    assert r == 3


def test_decode_query_token_limits(lib):
    """Q_S new tokens: 1..16, heads-per-KV-head x Q_S rows at most 64, and
    sparse_mode 0, 2 or 3 when Q_S > 1 (no MLA)."""
    q = t((2, 4, 3, 128))
    r, _ = decode_ws(lib, q, q, q, params(lib, num_heads=4, input_layout="BNSD", sparse_mode=3))
    assert r == 0
    q17 = t((2, 4, 17, 128))
    r, _ = decode_ws(lib, q17, q17, q17, params(lib, num_heads=4, input_layout="BNSD"))
    assert r == 5
    wide = t((2, 32, 3, 128))   # 32 heads on one KV head x 3 tokens = 96 rows
    kv = t((2, 1, 3, 128))
    r, _ = decode_ws(lib, wide, kv, kv, params(lib, num_heads=32, num_key_value_heads=1, input_layout="BNSD"))
    assert r == 5
    r, _ = decode_ws(lib, q, q, q, params(lib, num_heads=4, input_layout="BNSD", sparse_mode=4))
    assert r == 5
    qm = t((2, 2, 128, 512))
    lat = t((16, 128, 512))
    prm = params(lib, num_heads=128, num_key_value_heads=1, input_layout="BSND", block_size=128,
                 actual_seq_kvlen=[256])
    r, _ = decode_ws(lib, qm, lat, lat, prm, qr=t((2, 2, 128, 64)), kr=t((16, 128, 64)),
                     table=t((2, 2), B.DTYPE_I32))
    assert r == 5


def bsa_ws(lib, q, k, v, mask, shape, prm):
    ws = ctypes.c_size_t(0)
    s = (ctypes.c_int64 * 2)(*shape)
    m = ctypes.byref(mask) if mask is not None else None
    r = lib.bsa_get_workspace_size(ctypes.byref(q), ctypes.byref(k), ctypes.byref(v), m, s, ctypes.byref(prm.p),
                                   ctypes.byref(q), None, ctypes.byref(ws))
    return r, ws.value


def test_bsa_rules(lib):
    """aclnnBlockSparseAttentionV2 constraints: D in {64,128}; blockShapeY a
    multiple of 128; mask shape (B, N1, ceil(S/X), ceil(S/Y)); both length
    lists or neither; N1 % N2 == 0."""
    q, k = t((2, 8, 1000, 128)), t((2, 2, 1000, 128))
    good_mask = t((2, 8, 8, 8), B.DTYPE_U8)
    prm = params(lib, num_heads=8, num_key_value_heads=2, input_layout="BNSD")
    assert bsa_ws(lib, q, k, k, good_mask, (128, 128), prm)[0] == 0
    assert bsa_ws(lib, q, k, k, good_mask, (128, 100), prm)[0] == 3
    assert bsa_ws(lib, q, k, k, t((2, 8, 8, 7), B.DTYPE_U8), (128, 128), prm)[0] == 3
    assert bsa_ws(lib, q, k, k, good_mask, (128, 128), params(lib, num_heads=8, num_key_value_heads=2,
                                                               input_layout="BNSD", actual_seq_qlen=[5]))[0] == 6
    k3 = t((2, 3, 1000, 128))
    assert bsa_ws(lib, q, k3, k3, good_mask, (128, 128), params(lib, num_heads=8, num_key_value_heads=3,
                                                                 input_layout="BNSD"))[0] == 11
    q96 = t((2, 8, 1000, 96))
    assert bsa_ws(lib, q96, q96, q96, good_mask, (128, 128), params(lib, num_heads=8, input_layout="BNSD"))[0] == 5
    assert bsa_ws(lib, q, k, k, good_mask, (64, 128), prm)[0] == 5      # X not a multiple of 128 (library limit)
    assert bsa_ws(lib, q, k, k, None, (128, 128), prm)[0] == 1          # the bf16 entry needs its mask


def test_binding_fails_loudly_without_library(tmp_path):
    with pytest.raises(ImportError):
        B.load_library(str(tmp_path / "missing.so"))

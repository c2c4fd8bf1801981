"""Checks that pin the fp64 oracle to things other than itself.

Each check takes an oracle module (normally oracle.fia_oracle) so that the
mutation tests can run the same checks against deliberately broken copies and
show that every plausible mistake trips at least one of them.

Sources of truth used here:
  * a library routine: torch.nn.functional.scaled_dot_product_attention in
    float64 on the CPU, and scipy.special.logsumexp for the LSE;
  * closed forms of softmax attention (one allowed key, equal keys, zero keys,
    constant values) that need no attention code at all;
  * invariants the pages imply (paged == contiguous, GQA == repeated heads,
    TND == per-sequence calls, BSA all-ones == dense, LSE merge == unsplit);
  * the pages' empty-tensor rule (npu_fused_infer_attention_score_v2, "入参为空
    的处理"; aclnnFusedInferAttentionScoreV5, "公共约束"): K/V with S2 = 0 give
    attention_out = 0 and softmax_lse = +inf.
"""
from __future__ import annotations

import math

import numpy as np
import torch
from scipy.special import logsumexp

ATOL = 1e-10


def _rand(shape, seed):
    return torch.from_numpy(np.random.default_rng(seed).standard_normal(shape)).to(torch.float64)


def _sdpa(q, k, v, allowed, scale):
    """Library attention: q (n,d), k (m,d), v (m,dv), allowed (n,m) bool."""
    qt, kt, vt = (torch.as_tensor(np.asarray(x)).reshape(1, 1, *np.asarray(x).shape) for x in (q, k, v))
    out = torch.nn.functional.scaled_dot_product_attention(
        qt, kt, vt, attn_mask=torch.as_tensor(allowed).reshape(1, 1, *allowed.shape), scale=scale)
    return out[0, 0].numpy()


# -------------------------------------------------------------------- library
def check_rows_vs_library(orc):
    for seed, (n, m, d, dv) in enumerate([(5, 7, 4, 3), (9, 9, 8, 8), (3, 11, 6, 2)]):
        q, k, v = (_rand(s, 10 * seed + t).numpy() for t, s in enumerate([(n, d), (m, d), (m, dv)]))
        allowed = np.random.default_rng(seed + 99).random((n, m)) < 0.7
        allowed[:, 0] = True
        scale = 0.37 + seed
        out, lse = orc.attention_rows(q, k, v, allowed, scale)
        ref = _sdpa(q, k, v, allowed, scale)
        assert np.allclose(out, ref, atol=ATOL), "out != library softmax attention"
        s = scale * (q @ k.T)
        ref_lse = logsumexp(np.where(allowed, s, -np.inf), axis=1)
        assert np.allclose(lse, ref_lse, atol=ATOL), "lse != library logsumexp"


def check_prefill_causal_vs_library(orc):
    """sparse_mode 2 (top-left causal) equals the library's is_causal path."""
    B, N, S, D = 2, 3, 9, 8
    q, k, v = _rand((B, N, S, D), 1), _rand((B, N, S, D), 2), _rand((B, N, S, D), 3)
    out, _ = orc.fia_prefill(q, k, v, num_heads=N, scale_value=0.3, input_layout="BNSD", sparse_mode=2)
    ref = torch.nn.functional.scaled_dot_product_attention(q, k, v, is_causal=True, scale=0.3).numpy()
    assert np.allclose(out, ref, atol=ATOL), "mode 2 != library causal attention"


def check_gqa_vs_library(orc):
    """GQA with contiguous head groups equals the library's enable_gqa path
    (query head h uses key/value head h // (N1 / N2))."""
    B, N1, N2, S, D = 1, 6, 2, 5, 4
    q, k, v = _rand((B, N1, S, D), 4), _rand((B, N2, S, D), 5), _rand((B, N2, S, D), 6)
    out, _ = orc.fia_prefill(q, k, v, num_heads=N1, num_key_value_heads=N2, scale_value=0.5, input_layout="BNSD")
    kk = k.repeat_interleave(N1 // N2, dim=1)
    vv = v.repeat_interleave(N1 // N2, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, scale=0.5).numpy()
    assert np.allclose(out, ref, atol=ATOL), "GQA head grouping != repeat_interleave"


# --------------------------------------------------------------- closed forms
def check_closed_forms(orc):
    # (a) one allowed key: out = v_j, lse = s_j (here q . k_j = 2 * 3 on one axis)
    q = np.zeros((1, 4)); q[0, 1] = 2.0
    k = np.zeros((3, 4)); k[2, 1] = 3.0; k[0, 0] = 5.0
    v = np.arange(9, dtype=np.float64).reshape(3, 3)
    allowed = np.array([[False, False, True]])
    out, lse = orc.attention_rows(q, k, v, allowed, 0.5)
    assert np.allclose(out[0], v[2]) and abs(lse[0] - 3.0) < ATOL, "single key closed form"
    # (b) equal keys: out = mean of v over the allowed set, lse = s + ln|A|
    k = np.tile(np.array([[1.0, -2.0, 0.5, 0.0]]), (5, 1))
    q = np.array([[0.5, 0.25, 2.0, 7.0]])
    v = np.random.default_rng(0).standard_normal((5, 2))
    allowed = np.array([[True, False, True, True, False]])
    out, lse = orc.attention_rows(q, k, v, allowed, 1.0)
    s = 0.5 * 1.0 + 0.25 * -2.0 + 2.0 * 0.5
    assert np.allclose(out[0], v[[0, 2, 3]].mean(axis=0)), "equal keys -> mean"
    assert abs(lse[0] - (s + math.log(3))) < ATOL, "equal keys -> s + ln|A|"
    # (c) constant value rows give that constant for any scores
    q, k = _rand((4, 3), 7).numpy(), _rand((6, 3), 8).numpy()
    v = np.full((6, 2), -1.25)
    out, _ = orc.attention_rows(q, k, v, np.ones((4, 6), bool), 2.0)
    assert np.allclose(out, -1.25), "constant V"
    # (d) a row with no allowed key: out 0, lse +inf
    out, lse = orc.attention_rows(q, k, v, np.zeros((4, 6), bool), 2.0)
    assert np.all(out == 0) and np.all(np.isinf(lse) & (lse > 0)), "empty row -> 0 / +inf"


def check_mask_modes_by_counting(orc):
    """With K = 0 every allowed score is 0, so lse_i = ln(#allowed keys of row i)
    and, with V = identity, out_i is the uniform distribution over them.  This
    pins which keys each sparse_mode allows without re-deriving the rule."""
    def run(Sq, Skv, mode, mask=None, pre=2147483647, nxt=2147483647):
        q = _rand((1, 1, Sq, 4), 11)
        k = torch.zeros((1, 1, Skv, 4), dtype=torch.float64)
        v = torch.eye(Skv, dtype=torch.float64).reshape(1, 1, Skv, Skv)
        out, lse = orc.fia_prefill(q, k, v, num_heads=1, scale_value=1.0, input_layout="BNSD",
                                   sparse_mode=mode, atten_mask=mask, pre_tokens=pre, next_tokens=nxt)
        return out[0, 0], lse[0, 0, :, 0]

    # mode 2, leftUpCausal: row i sees keys 0..i
    out, lse = run(4, 6, 2)
    for i in range(4):
        assert abs(lse[i] - math.log(i + 1)) < ATOL, "mode 2 count"
        want = np.zeros(6); want[:i + 1] = 1.0 / (i + 1)
        assert np.allclose(out[i], want), "mode 2 set"
    # mode 3, rightDownCausal: row i sees keys 0..i + Skv - Sq
    out, lse = run(4, 6, 3)
    for i in range(4):
        assert abs(lse[i] - math.log(i + 3)) < ATOL, "mode 3 count"
        want = np.zeros(6); want[:i + 3] = 1.0 / (i + 3)
        assert np.allclose(out[i], want), "mode 3 set"
    # mode 4, band around the bottom-right diagonal: keys i+2-pre .. i+2+next
    out, lse = run(4, 6, 4, pre=1, nxt=0)
    for i in range(4):
        lo, hi = max(0, i + 2 - 1), min(5, i + 2)
        want = np.zeros(6); want[lo:hi + 1] = 1.0 / (hi - lo + 1)
        assert np.allclose(out[i], want), "mode 4 set"
    # mode 1 / mode 0 with an explicit mask: nonzero masks the pair
    mask = np.zeros((4, 6), dtype=np.uint8)
    mask[1, 3] = 1; mask[2, :5] = 1; mask[3, :] = 1
    out, lse = run(4, 6, 1, mask=mask)
    assert np.allclose(out[0], np.full(6, 1 / 6)), "mask row 0"
    want = np.full(6, 1 / 5); want[3] = 0
    assert np.allclose(out[1], want), "mask row 1"
    want = np.zeros(6); want[5] = 1
    assert np.allclose(out[2], want) and abs(lse[2]) < ATOL, "mask row 2"
    assert np.all(out[3] == 0) and lse[3] == np.inf, "fully masked row -> 0 / +inf"
    # mode 0 with mask and pre/next window (top-left anchored)
    out, lse = run(4, 6, 0, mask=np.zeros((4, 6), np.uint8), pre=1, nxt=1)
    for i in range(4):
        lo, hi = max(0, i - 1), min(5, i + 1)
        assert abs(lse[i] - math.log(hi - lo + 1)) < ATOL, "mode 0 window"


def check_mask_shapes_by_counting(orc):
    """atten_mask given per batch: the shapes (B,S1,S2) and (B,1,S1,S2) hold
    one mask per batch, (1,S1,S2) and (1,1,S1,S2) one mask for all
    (npu_fused_infer_attention_score_v2 / npu_prompt_flash_attention, parameter
    atten_mask).  With K = 0 and V = identity, row i of batch b attends
    uniformly to exactly the keys its own batch's mask leaves at 0, and
    lse = ln(count): each batch's counts are set by hand below, different per
    batch, so reading the wrong batch's mask changes the result."""
    B, Sq, Skv = 3, 4, 6
    q = _rand((B, 1, Sq, 4), 12)
    k = torch.zeros((B, 1, Skv, 4), dtype=torch.float64)
    v = torch.eye(Skv, dtype=torch.float64).reshape(1, 1, Skv, Skv).repeat(B, 1, 1, 1)
    # batch b, row i: keys 0 .. (b + i) % Skv visible, the rest masked
    per_batch = np.ones((B, Sq, Skv), dtype=np.uint8)
    for b in range(B):
        for i in range(Sq):
            per_batch[b, i, :(b + i) % Skv + 1] = 0
    forms = {"(B,S1,S2)": per_batch, "(B,1,S1,S2)": per_batch[:, None]}
    for name, mask in forms.items():
        out, lse = orc.fia_prefill(q, k, v, num_heads=1, scale_value=1.0, input_layout="BNSD", sparse_mode=1,
                                   atten_mask=mask)
        for b in range(B):
            for i in range(Sq):
                n = (b + i) % Skv + 1
                want = np.zeros(Skv); want[:n] = 1.0 / n
                assert np.allclose(out[b, 0, i], want, atol=ATOL), f"mask {name}: batch {b} row {i} set"
                assert abs(lse[b, 0, i, 0] - math.log(n)) < ATOL, f"mask {name}: batch {b} row {i} count"
    # one mask shared by every batch: batch 1's pattern for all
    for name, mask in {"(1,S1,S2)": per_batch[1:2], "(1,1,S1,S2)": per_batch[1:2, None]}.items():
        out, lse = orc.fia_prefill(q, k, v, num_heads=1, scale_value=1.0, input_layout="BNSD", sparse_mode=1,
                                   atten_mask=mask)
        for b in range(B):
            for i in range(Sq):
                n = (1 + i) % Skv + 1
                assert abs(lse[b, 0, i, 0] - math.log(n)) < ATOL, f"mask {name}: broadcast to batch {b}"
    # TND with a per-batch mask: rows and keys are batch-local
    lens = [2, 4, 3]
    cum = list(np.cumsum(lens))
    qt = _rand((sum(lens), 1, 4), 13)
    kt = torch.zeros((sum(lens), 1, 4), dtype=torch.float64)
    vt = torch.eye(sum(lens), dtype=torch.float64)[:, None, :]
    out, lse = orc.fia_prefill(qt, kt, vt, num_heads=1, scale_value=1.0, input_layout="TND", sparse_mode=1,
                               atten_mask=per_batch, actual_seq_qlen=cum, actual_seq_kvlen=cum)
    start = 0
    for b, L in enumerate(lens):
        for i in range(L):
            n = min((b + i) % Skv + 1, L)
            want = np.zeros(sum(lens)); want[start:start + n] = 1.0 / n
            assert np.allclose(out[start + i, 0], want, atol=ATOL), f"TND mask batch {b} row {i}"
        start += L


def check_decode_mask_by_counting(orc):
    """Decode atten_mask (B, KV_S), also as (B,1,KV_S) / (B,1,1,KV_S), one row
    of keys per batch; (1, KV_S) is shared (npu_fused_infer_attention_score_v2,
    atten_mask for Q_S = 1).  K = 0, V = identity: out is uniform over the
    batch's unmasked keys and lse = ln(count), counts set by hand per batch."""
    B, N, Skv = 3, 2, 5
    q = _rand((B, N, 1, 4), 14)
    k = torch.zeros((B, N, Skv, 4), dtype=torch.float64)
    v = torch.eye(Skv, dtype=torch.float64).reshape(1, 1, Skv, Skv).repeat(B, N, 1, 1)
    m = np.zeros((B, Skv), dtype=np.uint8)
    m[0, 1] = 1                  # batch 0: keys {0, 2, 3, 4}
    m[1, :3] = 1                 # batch 1: keys {3, 4}
    m[2, [0, 2, 4]] = 1          # batch 2: keys {1, 3}
    visible = [[0, 2, 3, 4], [3, 4], [1, 3]]
    for name, mask in {"(B,KV_S)": m, "(B,1,KV_S)": m[:, None], "(B,1,1,KV_S)": m[:, None, None]}.items():
        out, lse = orc.fia_decode(q, k, v, num_heads=N, input_layout="BNSD", atten_mask=mask)
        for b in range(B):
            want = np.zeros(Skv); want[visible[b]] = 1.0 / len(visible[b])
            for h in range(N):
                assert np.allclose(out[b, h, 0], want, atol=ATOL), f"decode mask {name}: batch {b}"
                assert abs(lse[b, h, 0, 0] - math.log(len(visible[b]))) < ATOL, f"decode mask {name}: count"
    out, lse = orc.fia_decode(q, k, v, num_heads=N, input_layout="BNSD", atten_mask=m[1:2])
    for b in range(B):
        assert abs(lse[b, 0, 0, 0] - math.log(2)) < ATOL, "decode mask (1, KV_S) broadcast"


def check_softmax_rows_sum_to_one(orc):
    """With V = identity the output rows are the softmax probabilities."""
    q, k = _rand((1, 2, 5, 3), 20), _rand((1, 2, 7, 3), 21)
    v = torch.eye(7, dtype=torch.float64).reshape(1, 1, 7, 7).repeat(1, 2, 1, 1)
    out, _ = orc.fia_prefill(q, k, v, num_heads=2, scale_value=1.3, input_layout="BNSD")
    assert np.allclose(out.sum(axis=-1), 1.0, atol=1e-12) and np.all(out >= 0), "rows sum to 1"


# ----------------------------------------------------------------- invariants
def check_layouts_agree(orc):
    B, N, S, D = 2, 2, 5, 4
    q, k, v = _rand((B, N, S, D), 30), _rand((B, N, S, D), 31), _rand((B, N, S, D), 32)
    ref, lref = orc.fia_prefill(q, k, v, num_heads=N, scale_value=0.7, input_layout="BNSD", sparse_mode=2)
    t = lambda x: x.transpose(1, 2).contiguous()
    o2, l2 = orc.fia_prefill(t(q), t(k), t(v), num_heads=N, scale_value=0.7, input_layout="BSND", sparse_mode=2)
    assert np.allclose(o2.transpose(0, 2, 1, 3), ref, atol=ATOL) and np.allclose(l2, lref), "BSND"
    h = lambda x: t(x).reshape(B, S, N * D)
    o3, _ = orc.fia_prefill(h(q), h(k), h(v), num_heads=N, scale_value=0.7, input_layout="BSH", sparse_mode=2)
    assert np.allclose(o3.reshape(B, S, N, D).transpose(0, 2, 1, 3), ref, atol=ATOL), "BSH"


def check_tnd_equals_per_sequence(orc):
    lens = [3, 1, 6]
    N1, N2, D = 4, 2, 4
    T = sum(lens)
    q, k, v = _rand((T, N1, D), 40), _rand((T, N2, D), 41), _rand((T, N2, D), 42)
    cum = list(np.cumsum(lens))
    out, lse = orc.fia_prefill(q, k, v, num_heads=N1, num_key_value_heads=N2, scale_value=0.5,
                               input_layout="TND", sparse_mode=3, actual_seq_qlen=cum, actual_seq_kvlen=cum)
    s = 0
    for L in lens:
        sl = slice(s, s + L)
        o, l = orc.fia_prefill(q[sl].permute(1, 0, 2)[None], k[sl].permute(1, 0, 2)[None],
                               v[sl].permute(1, 0, 2)[None], num_heads=N1, num_key_value_heads=N2,
                               scale_value=0.5, input_layout="BNSD", sparse_mode=3)
        assert np.allclose(out[sl], o[0].transpose(1, 0, 2), atol=ATOL), "TND out"
        assert np.allclose(lse[sl, :, 0], l[0, :, :, 0].T, atol=ATOL), "TND lse"
        s += L


def check_actual_lengths_equal_truncation(orc):
    """actual_seq lengths behave as slicing the tensors; rows past the query
    length are padding (0 / +inf)."""
    q, k, v = _rand((2, 2, 6, 4), 50), _rand((2, 2, 7, 4), 51), _rand((2, 2, 7, 4), 52)
    out, lse = orc.fia_prefill(q, k, v, num_heads=2, scale_value=0.5, input_layout="BNSD",
                               actual_seq_qlen=[4, 6], actual_seq_kvlen=[5])
    for b, (lq, lk) in enumerate([(4, 5), (6, 5)]):
        o, l = orc.fia_prefill(q[b:b + 1, :, :lq], k[b:b + 1, :, :lk], v[b:b + 1, :, :lk], num_heads=2,
                               scale_value=0.5, input_layout="BNSD")
        assert np.allclose(out[b, :, :lq], o[0], atol=ATOL) and np.allclose(lse[b, :, :lq], l[0]), "actual lengths"
        assert np.all(out[b, :, lq:] == 0) and np.all(np.isinf(lse[b, :, lq:])), "padding rows"


def check_paged_equals_contiguous(orc):
    """Scatter a contiguous cache into a shuffled block pool; the paged gather
    must give back exactly the contiguous result."""
    B, N1, N2, D, bs = 3, 4, 2, 8, 4
    lens = [9, 4, 1]
    S = 12
    rng = np.random.default_rng(7)
    q = _rand((B, N1, 1, D), 60)
    k, v = _rand((B, N2, S, D), 61), _rand((B, N2, S, D), 62)
    nblk = B * (S // bs)
    perm = rng.permutation(nblk)
    table = perm.reshape(B, S // bs).astype(np.int32)
    kp = torch.zeros((nblk, N2, bs, D), dtype=torch.float64)
    vp = torch.zeros_like(kp)
    kh = torch.zeros((nblk, bs, N2 * D), dtype=torch.float64)
    vh = torch.zeros_like(kh)
    for b in range(B):
        for i in range(S // bs):
            kp[table[b, i]] = k[b, :, i * bs:(i + 1) * bs]
            vp[table[b, i]] = v[b, :, i * bs:(i + 1) * bs]
            kh[table[b, i]] = k[b, :, i * bs:(i + 1) * bs].permute(1, 0, 2).reshape(bs, N2 * D)
            vh[table[b, i]] = v[b, :, i * bs:(i + 1) * bs].permute(1, 0, 2).reshape(bs, N2 * D)
    ref, lref = orc.fia_decode(q, k, v, num_heads=N1, num_key_value_heads=N2, scale_value=0.4,
                               input_layout="BNSD", actual_seq_kvlen=lens)
    for pk, pv in ((kp, vp), (kh, vh)):
        out, lse = orc.fia_decode(q, pk, pv, num_heads=N1, num_key_value_heads=N2, scale_value=0.4,
                                  input_layout="BNSD", actual_seq_kvlen=lens, block_table=table, block_size=bs)
        assert np.array_equal(out, ref) and np.array_equal(lse, lref), "paged != contiguous"


def check_decode_equals_prefill_row(orc):
    q, k, v = _rand((2, 4, 1, 8), 70), _rand((2, 2, 9, 8), 71), _rand((2, 2, 9, 8), 72)
    o1, l1 = orc.fia_decode(q, k, v, num_heads=4, num_key_value_heads=2, scale_value=0.3, input_layout="BNSD",
                            actual_seq_kvlen=[9, 3])
    o2, l2 = orc.fia_prefill(q, k, v, num_heads=4, num_key_value_heads=2, scale_value=0.3, input_layout="BNSD",
                             actual_seq_kvlen=[9, 3])
    assert np.allclose(o1, o2, atol=ATOL) and np.allclose(l1, l2, atol=ATOL), "decode == one-row prefill"


def check_multitoken_decode_vs_library(orc):
    """Q_S new tokens against a paged cache, right-down causal (sparse_mode 3):
    token t of a sequence of L keys sees keys 0 .. L - Q_S + t.  Reference: the
    cache gathered here by hand and the library's attention with that mask;
    mode 0 lets every token see the whole cache."""
    B, N1, N2, QS, D, bs = 2, 4, 2, 3, 8, 4
    lens = [10, 2]
    nblk = 6
    kp, vp = _rand((nblk, N2, bs, D), 90), _rand((nblk, N2, bs, D), 91)
    table = np.array([[4, 1, 5], [0, 2, 3]], dtype=np.int32)
    q = _rand((B, N1, QS, D), 92)
    for mode in (3, 0):
        out, lse = orc.fia_decode(q, kp, vp, num_heads=N1, num_key_value_heads=N2, scale_value=0.35,
                                  input_layout="BNSD", actual_seq_kvlen=lens, block_table=table, block_size=bs,
                                  sparse_mode=mode)
        assert out.shape == (B, N1, QS, D) and lse.shape == (B, N1, QS, 1)
        for b in range(B):
            L = lens[b]
            for h in range(N1):
                kv = h // (N1 // N2)
                kk = torch.stack([kp[table[b, j // bs], kv, j % bs] for j in range(L)])
                vv = torch.stack([vp[table[b, j // bs], kv, j % bs] for j in range(L)])
                allowed = np.array([[mode == 0 or j <= L - QS + t for j in range(L)] for t in range(QS)])
                live = allowed.any(axis=1)
                ref = _sdpa(q[b, h].numpy()[live], kk.numpy(), vv.numpy(), allowed[live], 0.35)
                assert np.allclose(out[b, h][live], ref, atol=ATOL), "multi-token decode != library attention"
                s = 0.35 * (q[b, h].numpy() @ kk.numpy().T)
                ref_lse = logsumexp(np.where(allowed[live], s[live], -np.inf), axis=1)
                assert np.allclose(lse[b, h, live, 0], ref_lse, atol=ATOL), "multi-token lse"
                assert np.all(out[b, h][~live] == 0) and np.all(np.isinf(lse[b, h, ~live, 0])), "tokens with no key"


def check_paged_prefill_equals_contiguous(orc):
    """Chunked prefill against a paged cache equals prefill over the contiguous
    keys the pages scatter: the pool here is filled by hand (logical block i of
    batch b goes to physical block perm[...], row r of it = key i * bs + r), in
    both cache layouts, for a padded and a TND query, causal and band masks."""
    B, N1, N2, D, bs = 2, 4, 2, 8, 4
    lens_q, lens_kv = [3, 5], [9, 6]
    S = max(lens_kv)
    k, v = _rand((B, N2, S, D), 130), _rand((B, N2, S, D), 131)
    perm = [5, 1, 3, 0, 4]          # physical block of each (batch, logical block), in order
    nblk = 7
    table = np.full((B, 3), 6, dtype=np.int32)
    pools = {"BNBD": (torch.full((nblk, N2, bs, D), float("nan"), dtype=torch.float64),
                      torch.full((nblk, N2, bs, D), float("nan"), dtype=torch.float64)),
             "BBH": (torch.full((nblk, bs, N2 * D), float("nan"), dtype=torch.float64),
                     torch.full((nblk, bs, N2 * D), float("nan"), dtype=torch.float64))}
    pos = 0
    for b in range(B):
        for i in range(-(-lens_kv[b] // bs)):
            blk = perm[pos]; pos += 1
            table[b, i] = blk
            for r in range(bs):
                j = i * bs + r
                if j >= lens_kv[b]:
                    continue
                pools["BNBD"][0][blk, :, r] = k[b, :, j]; pools["BNBD"][1][blk, :, r] = v[b, :, j]
                pools["BBH"][0][blk, r] = k[b, :, j].reshape(-1); pools["BBH"][1][blk, r] = v[b, :, j].reshape(-1)
    q = _rand((B, N1, max(lens_q), D), 132)
    for layout_kv, (kp, vp) in pools.items():
        for mode, extra in ((3, {}), (4, {"pre_tokens": 2, "next_tokens": 0}), (2, {})):
            want_o, want_l = orc.fia_prefill(q, k, v, num_heads=N1, num_key_value_heads=N2, scale_value=0.4,
                                             input_layout="BNSD", sparse_mode=mode, actual_seq_qlen=lens_q,
                                             actual_seq_kvlen=lens_kv, **extra)
            got_o, got_l = orc.fia_prefill_paged(q, kp, vp, block_table=table, block_size=bs,
                                                 actual_seq_kvlen=lens_kv, num_heads=N1, num_key_value_heads=N2,
                                                 scale_value=0.4, input_layout="BNSD", sparse_mode=mode,
                                                 actual_seq_qlen=lens_q, **extra)
            assert np.array_equal(got_o, want_o) and np.array_equal(got_l, want_l), "paged prefill != contiguous"
        # TND query: rows of both sequences packed, kv lengths per batch
        qt = torch.cat([q[b, :, :lens_q[b]].transpose(0, 1) for b in range(B)])
        got_o, got_l = orc.fia_prefill_paged(qt, kp, vp, block_table=table, block_size=bs, actual_seq_kvlen=lens_kv,
                                             num_heads=N1, num_key_value_heads=N2, scale_value=0.4,
                                             input_layout="TND", sparse_mode=3, actual_seq_qlen=[3, 8])
        want_o, want_l = orc.fia_prefill(q, k, v, num_heads=N1, num_key_value_heads=N2, scale_value=0.4,
                                         input_layout="BNSD", sparse_mode=3, actual_seq_qlen=lens_q,
                                         actual_seq_kvlen=lens_kv)
        for b, (s0, L) in enumerate(((0, 3), (3, 5))):
            assert np.array_equal(got_o[s0:s0 + L], want_o[b, :, :L].transpose(1, 0, 2)), "TND paged prefill"
            assert np.array_equal(got_l[s0:s0 + L, :, 0], want_l[b, :, :L, 0].T), "TND paged lse"


def check_mla_prefill_vs_library(orc):
    """MLA prefill: scores over [q, q_rope] . [k, k_rope], value with its own
    D.  Reference: the library's attention on the concatenation built here, per
    sequence and head of a TND batch (right-down causal); the BSH layout
    (rope concatenated per head) agrees with BNSD."""
    N1, N2, D, Dr, Dv = 4, 2, 8, 4, 6
    lq, lk = [3, 5], [4, 5]
    q, qr = _rand((8, N1, D), 140), _rand((8, N1, Dr), 141)
    k, kr, v = _rand((9, N2, D), 142), _rand((9, N2, Dr), 143), _rand((9, N2, Dv), 144)
    out, lse = orc.fia_prefill(q, k, v, query_rope=qr, key_rope=kr, num_heads=N1, num_key_value_heads=N2,
                               scale_value=0.3, input_layout="TND", sparse_mode=3, actual_seq_qlen=[3, 8],
                               actual_seq_kvlen=[4, 9])
    assert out.shape == (8, N1, Dv) and lse.shape == (8, N1, 1)
    for b, (q0, k0) in enumerate(((0, 0), (3, 4))):
        for h in range(N1):
            kv = h // (N1 // N2)
            qc = torch.cat([q[q0:q0 + lq[b], h], qr[q0:q0 + lq[b], h]], dim=1).numpy()
            kc = torch.cat([k[k0:k0 + lk[b], kv], kr[k0:k0 + lk[b], kv]], dim=1).numpy()
            vv = v[k0:k0 + lk[b], kv].numpy()
            allowed = np.array([[j <= i + lk[b] - lq[b] for j in range(lk[b])] for i in range(lq[b])])
            ref = _sdpa(qc, kc, vv, allowed, 0.3)
            assert np.allclose(out[q0:q0 + lq[b], h], ref, atol=ATOL), "MLA prefill != library attention"
            ref_lse = logsumexp(np.where(allowed, 0.3 * qc @ kc.T, -np.inf), axis=1)
            assert np.allclose(lse[q0:q0 + lq[b], h, 0], ref_lse, atol=ATOL), "MLA prefill lse"
    # BSH (heads packed in H) against BNSD
    qb, qrb = _rand((2, N1, 5, D), 145), _rand((2, N1, 5, Dr), 146)
    kb, krb, vb = _rand((2, N2, 6, D), 147), _rand((2, N2, 6, Dr), 148), _rand((2, N2, 6, Dv), 149)
    o1, l1 = orc.fia_prefill(qb, kb, vb, query_rope=qrb, key_rope=krb, num_heads=N1, num_key_value_heads=N2,
                             scale_value=0.3, input_layout="BNSD", sparse_mode=2)
    bsh = lambda x: x.transpose(1, 2).reshape(x.shape[0], x.shape[2], -1)
    o2, l2 = orc.fia_prefill(bsh(qb), bsh(kb), bsh(vb), query_rope=bsh(qrb), key_rope=bsh(krb), num_heads=N1,
                             num_key_value_heads=N2, scale_value=0.3, input_layout="BSH", sparse_mode=2)
    assert np.allclose(o2, bsh(torch.from_numpy(o1)).numpy(), atol=ATOL) and np.allclose(l1, l2, atol=ATOL), \
        "MLA prefill BSH != BNSD"


def check_mla_equals_concatenated_attention(orc):
    B, N1, Dl, Dr, bs = 2, 4, 16, 4, 4
    lens = [7, 8]
    nblk = 4
    lat, rope = _rand((nblk, bs, Dl), 80), _rand((nblk, bs, Dr), 81)
    table = np.array([[2, 0], [1, 3]], dtype=np.int32)
    q, qr = _rand((B, 1, N1, Dl), 82), _rand((B, 1, N1, Dr), 83)
    out, lse = orc.fia_decode(q, lat, lat, num_heads=N1, num_key_value_heads=1, scale_value=0.2,
                              input_layout="BSND", actual_seq_kvlen=lens, block_table=table, block_size=bs,
                              query_rope=qr, key_rope=rope)
    for b in range(B):
        kk = torch.cat([torch.cat([lat[table[b, j // bs], j % bs], rope[table[b, j // bs], j % bs]])[None]
                        for j in range(lens[b])])
        vv = torch.cat([lat[table[b, j // bs], j % bs][None] for j in range(lens[b])])
        qq = torch.cat([q[b, 0], qr[b, 0]], dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(qq[None], kk[None], vv[None], scale=0.2)[0].numpy()
        assert np.allclose(out[b, 0], ref, atol=ATOL), "MLA != attention over [latent, rope]"


def check_bsa(orc):
    B, N1, N2, S, D, X, Y = 1, 4, 2, 10, 4, 3, 4
    q, k, v = _rand((B, N1, S, D), 90), _rand((B, N2, S, D), 91), _rand((B, N2, S, D), 92)
    nq, nk = -(-S // X), -(-S // Y)
    ones = np.ones((B, N1, nq, nk), np.uint8)
    o1, l1 = orc.bsa_forward(q, k, v, ones, (X, Y), num_heads=N1, num_key_value_heads=N2, scale_value=0.5)
    o2, l2 = orc.fia_prefill(q, k, v, num_heads=N1, num_key_value_heads=N2, scale_value=0.5, input_layout="BNSD")
    assert np.allclose(o1, o2, atol=ATOL) and np.allclose(l1, l2, atol=ATOL), "BSA all-ones != dense"
    m = (np.random.default_rng(3).random((B, N1, nq, nk)) < 0.5).astype(np.uint8)
    m[:, :, :, 0] = 1
    o1, l1 = orc.bsa_forward(q, k, v, m, (X, Y), num_heads=N1, num_key_value_heads=N2, scale_value=0.5)
    for h in range(N1):
        expanded = np.kron(m[0, h], np.ones((X, Y), np.uint8))[:S, :S]     # 1 = keep
        o2, l2 = orc.fia_prefill(q[:, h:h + 1], k[:, h // 2:h // 2 + 1], v[:, h // 2:h // 2 + 1], num_heads=1,
                                 scale_value=0.5, input_layout="BNSD", sparse_mode=1,
                                 atten_mask=(1 - expanded))
        assert np.allclose(o1[:, h:h + 1], o2, atol=ATOL) and np.allclose(l1[:, h:h + 1], l2), "BSA != expanded mask"


def check_bsa_fp8_dequant(orc):
    """FP8 block-sparse attention: dequant scales per block of X query rows and
    Y key / value rows.  (a) A query block whose scale is 0 has all scores 0:
    each of its rows is the plain mean of the dequantised value rows it may see
    (closed form), and the rows of the other query block do not change.
    (b) Output is linear in the value scales.  (c) Only the product of query
    and key scales enters the scores.  (d) With unit scales the result is the
    bf16 path's on the same values (e4m3 values are exact in bf16)."""
    B, N1, N2, S, D, X, Y = 1, 2, 1, 10, 4, 4, 6
    g = torch.Generator().manual_seed(150)
    f8 = lambda shape: (torch.randn(shape, generator=g, dtype=torch.float64) * 4).clamp(-448, 448).to(
        torch.float8_e4m3fn)
    q, k, v = f8((B, N1, S, D)), f8((B, N2, S, D)), f8((B, N2, S, D))
    nq, nk = -(-S // X), -(-S // Y)
    m = np.ones((B, N1, nq, nk), np.uint8)
    m[0, 1, 1, 1] = 0
    pos = lambda shape, seed: torch.rand(shape, generator=torch.Generator().manual_seed(seed),
                                         dtype=torch.float64) + 0.5
    qs, ks, vs = pos((B, N1, nq, 1), 151).float(), pos((B, N2, nk, 1), 152).float(), pos((B, N2, nk, 1), 153).float()
    run = lambda a, b, c: orc.bsa_forward(q, k, v, m, (X, Y), num_heads=N1, num_key_value_heads=N2, scale_value=0.3,
                                          q_dequant_scale=a, k_dequant_scale=b, v_dequant_scale=c)
    o, l = run(qs, ks, vs)
    qz = qs.clone()
    qz[0, :, 0] = 0
    oz, lz = run(qz, ks, vs)
    vdq = v.to(torch.float64).numpy()[0, 0] * np.repeat(vs.numpy()[0, 0, :, 0], Y)[:S, None]
    for h in range(N1):
        for i in range(X):
            keep = np.repeat(m[0, h, i // X], Y)[:S] != 0
            assert np.allclose(oz[0, h, i], vdq[keep].mean(axis=0), atol=1e-9), "zero query scale -> mean of V"
            assert abs(lz[0, h, i, 0] - math.log(keep.sum())) < 1e-9, "zero query scale -> lse = ln(count)"
    assert np.array_equal(oz[:, :, X:], o[:, :, X:]), "a query block's scale leaks into another block"
    o2, _ = run(qs, ks, vs * 2)
    assert np.allclose(o2, 2 * o, atol=1e-9), "output linear in the value scales"
    o3, l3 = run(qs * 4, ks / 4, vs)
    assert np.allclose(o3, o, atol=1e-9) and np.allclose(l3, l, atol=1e-9), "only q scale x k scale matters"
    ones_q, ones_k = torch.ones_like(qs), torch.ones_like(ks)
    o4, l4 = run(ones_q, ones_k, ones_k)
    o5, l5 = orc.bsa_forward(q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), m, (X, Y),
                             num_heads=N1, num_key_value_heads=N2, scale_value=0.3)
    assert np.array_equal(o4, o5) and np.array_equal(l4, l5), "unit scales != bf16 path"
    # TND: the same single sequence packed as (T, N, D) dequantises the same way
    tnd = lambda x: x[0].transpose(0, 1).contiguous()
    o6, l6 = orc.bsa_forward(tnd(q), tnd(k), tnd(v), m, (X, Y), num_heads=N1, num_key_value_heads=N2,
                             scale_value=0.3, input_layout="TND", actual_seq_qlen=[S], actual_seq_kvlen=[S],
                             q_dequant_scale=qs, k_dequant_scale=ks, v_dequant_scale=vs)
    assert np.allclose(o6, o[0].transpose(1, 0, 2), atol=1e-12) and np.allclose(l6[:, :, 0], l[0, :, :, 0].T), \
        "FP8 TND != BNSD"


def check_fp8_dense_vs_library(orc):
    """Dense FP8 attention (every block kept): the oracle equals library
    attention on the dequantised values, query row i scaled by its block's
    q scale, key / value row j by its block's k / v scale (GQA, ragged last
    blocks)."""
    B, N1, N2, S, D, X, Y = 1, 4, 2, 11, 8, 4, 6
    g = torch.Generator().manual_seed(160)
    f8 = lambda shape: (torch.randn(shape, generator=g, dtype=torch.float64) * 4).clamp(-448, 448).to(
        torch.float8_e4m3fn)
    q, k, v = f8((B, N1, S, D)), f8((B, N2, S, D)), f8((B, N2, S, D))
    nq, nk = -(-S // X), -(-S // Y)
    pos = lambda shape, seed: (torch.rand(shape, generator=torch.Generator().manual_seed(seed),
                                          dtype=torch.float64) + 0.5).float()
    qs, ks, vs = pos((B, N1, nq, 1), 161), pos((B, N2, nk, 1), 162), pos((B, N2, nk, 1), 163)
    m = np.ones((B, N1, nq, nk), np.uint8)
    o, l = orc.bsa_forward(q, k, v, m, (X, Y), num_heads=N1, num_key_value_heads=N2, scale_value=0.25,
                           q_dequant_scale=qs, k_dequant_scale=ks, v_dequant_scale=vs)
    grp = N1 // N2
    for h in range(N1):
        qd = q.to(torch.float64).numpy()[0, h] * np.repeat(qs.double().numpy()[0, h, :, 0], X)[:S, None]
        kd = k.to(torch.float64).numpy()[0, h // grp] * np.repeat(ks.double().numpy()[0, h // grp, :, 0], Y)[:S, None]
        vd = v.to(torch.float64).numpy()[0, h // grp] * np.repeat(vs.double().numpy()[0, h // grp, :, 0], Y)[:S, None]
        ref = _sdpa(qd, kd, vd, np.ones((S, S), bool), 0.25)
        assert np.allclose(o[0, h], ref, atol=1e-9), "dense FP8 != library attention on dequantised values"
        lref = logsumexp(0.25 * qd @ kd.T, axis=1)
        assert np.allclose(l[0, h, :, 0], lref, atol=1e-9), "dense FP8 lse"


def check_lse_merge(orc):
    """Split the keys in two, attend to each half, merge by LSE: equals unsplit."""
    q, k, v = _rand((6, 4), 100).numpy(), _rand((10, 4), 101).numpy(), _rand((10, 3), 102).numpy()
    allowed = np.ones((6, 10), bool)
    allowed[5] = False
    allowed[4, 6:] = False       # row 4 has keys only in the first half
    o, l = orc.attention_rows(q, k, v, allowed, 0.8)
    oa, la = orc.attention_rows(q, k[:6], v[:6], allowed[:, :6], 0.8)
    ob, lb = orc.attention_rows(q, k[6:], v[6:], allowed[:, 6:], 0.8)
    om, lm = orc.lse_merge([oa, ob], [la, lb])
    assert np.allclose(om, o, atol=ATOL) and np.allclose(lm, l, atol=ATOL), "LSE merge"


def check_empty_rules(orc):
    """K/V with S2 = 0: out all zeros, lse all +inf (pages' empty-tensor rule)."""
    q = _rand((1, 2, 3, 4), 110)
    k = torch.zeros((1, 2, 0, 4), dtype=torch.float64)
    out, lse = orc.fia_prefill(q, k, k, num_heads=2, scale_value=1.0, input_layout="BNSD")
    assert out.shape == (1, 2, 3, 4) and np.all(out == 0) and np.all(lse == np.inf), "empty KV"
    out, lse = orc.fia_decode(q[:, :, :1], k, k, num_heads=2, input_layout="BNSD")
    assert np.all(out == 0) and np.all(lse == np.inf), "empty KV decode"


ALL_CHECKS = [
    check_rows_vs_library, check_prefill_causal_vs_library, check_gqa_vs_library, check_closed_forms,
    check_mask_modes_by_counting, check_mask_shapes_by_counting, check_decode_mask_by_counting,
    check_softmax_rows_sum_to_one, check_layouts_agree,
    check_tnd_equals_per_sequence, check_actual_lengths_equal_truncation, check_paged_equals_contiguous,
    check_decode_equals_prefill_row, check_multitoken_decode_vs_library, check_paged_prefill_equals_contiguous,
    check_mla_prefill_vs_library, check_mla_equals_concatenated_attention,
    check_bsa, check_bsa_fp8_dequant, check_fp8_dense_vs_library, check_lse_merge,
    check_empty_rules,
]

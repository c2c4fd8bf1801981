"""Plain fp64 CPU oracle for fused inference attention.

TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the benchmark's
CPU-baseline / reference legs may import this module.  The CUDA library never
does, and this module imports nothing from it.

What it computes is the plain definition the pages give, written out step by
step with numpy float64 (matrix products are the only library primitive used):

  attention_out = softmax(scale * Q K^T + atten_mask) V
      -- torch_npu.npu_prompt_flash_attention, "功能说明" (formula);
         torch_npu.npu_fused_infer_attention_score_v2, "计算公式";
         aclnnBlockSparseAttentionV2, "计算公式" (key/value restricted to the
         blocks blockSparseMask selects).
  softmax_lse = log(sum(exp(s - max(s)))) + max(s)
      -- npu_fused_infer_attention_score_v2, output "softmax_lse": take the max
         of Q K^T, subtract it, exponentiate, sum, take the log, add the max back.

Inputs arrive as torch tensors already rounded to fp16/bf16 and are upcast
exactly to float64.  Outputs are float64 numpy arrays.

Readings taken where the pages are silent, garbled or contradict each other:
  * GQA: query head h reads key/value head floor(h / (Q_N / KV_N)).
  * atten_mask: a nonzero / True element masks the pair (adds -inf).
  * sparse_mode 2: key j is allowed for query i iff j <= i (top-left aligned);
    sparse_mode 3: j <= i + S_kv - S_q (bottom-right aligned);
    sparse_mode 4: i + S_kv - S_q - pre_tokens <= j <= i + S_kv - S_q + next_tokens;
    sparse_mode 0 with a mask: mask[i, j] == 0 and i - pre_tokens <= j <= i + next_tokens;
    sparse_mode 0 without a mask: all keys; sparse_mode 1: the mask alone.
    Modes 2/3/4 are computed from indices; the compressed 2048x2048 mask
    tensor those modes take on Ascend is not read.
  * A query row with no allowed key (empty K/V, a fully masked row, or a
    padding row past the batch's actual length) gets out = 0 and lse = +inf,
    extending the pages' empty-tensor rule to single rows.
  * TND: actual_seq_* are cumulative sums without a leading 0; B is the list length.
  * MLA: scores = scale * (q.k + q_rope.k_rope) over the 576-dim concatenation;
    the value is the 512-d latent.
  * blockSparseMask: nonzero keeps the (X x Y) block; head index is the query head.
  * MLA prefill: the score is scale * (q.k + q_rope.k_rope), as for MLA decode.
  * Prefill against a paged cache: actual_seq_kvlen holds per-batch key
    counts, also for a TND query (the cache is paged, not packed).
  * FP8 block-sparse: query rows dequantised per X-row block, key / value rows
    per Y-row block (X = 128, Y = 256 or 512 on the pages).

Parity is pinned by tests/test_oracle_pins.py (closed forms, a library softmax
attention, invariants and the pages' empty-tensor rule).  No numeric output
printed on the pages is reproducible (the worked example draws unseeded random
inputs), so no function here is pinned to a printed value.
"""
from __future__ import annotations

import numpy as np

INT32_MAX = 2147483647


def f64(t) -> np.ndarray:
    """Exact upcast of an fp16/bf16/fp32 torch tensor (or array) to float64."""
    if hasattr(t, "detach"):
        import torch
        return t.detach().cpu().to(torch.float64).numpy()
    return np.asarray(t, dtype=np.float64)


# ---------------------------------------------------------------------------
# Step 1: per-batch lengths
#   npu_fused_infer_attention_score_v2, parameters actual_seq_qlen / actual_seq_kvlen:
#   absent -> the tensor's S; a list of length 1 is used for every batch; a list
#   of length >= B contributes its first B entries; any other length is an error;
#   each entry must not exceed the tensor's S.  For TND every entry is the sum
#   of this batch's length and all earlier ones, so B = len(list).
# ---------------------------------------------------------------------------
def resolve_lengths(lst, B: int, S: int) -> list[int]:
    if lst is None:
        return [S] * B
    lst = [int(x) for x in lst]
    if len(lst) == 1:
        lens = lst * B
    elif len(lst) >= B:
        lens = lst[:B]
    else:
        raise ValueError("actual_seq length list must have 1 or >= B entries")
    for n in lens:
        if n < 0 or n > S:
            raise ValueError("actual_seq entry out of range")
    return lens


def tnd_lengths(cum) -> tuple[list[int], list[int]]:
    """Cumulative list (no leading 0) -> (starts, lengths)."""
    starts, lens, prev = [], [], 0
    for c in cum:
        c = int(c)
        if c < prev:
            raise ValueError("TND cumulative lengths must be non-decreasing")
        starts.append(prev)
        lens.append(c - prev)
        prev = c
    return starts, lens


# ---------------------------------------------------------------------------
# Step 2: the allowed key set of every query row (the atten_mask term)
#   sparse_mode semantics: npu_fused_infer_attention_score_v2, parameter
#   sparse_mode; npu_prompt_flash_attention, parameters atten_mask, sparse_mode.
# ---------------------------------------------------------------------------
def allowed_matrix(Sq: int, Skv: int, sparse_mode: int = 0, mask2d=None,
                   pre_tokens: int = INT32_MAX, next_tokens: int = INT32_MAX) -> np.ndarray:
    i = np.arange(Sq)[:, None]
    j = np.arange(Skv)[None, :]
    if sparse_mode == 0:
        if mask2d is None:
            ok = np.ones((Sq, Skv), dtype=bool)
        else:
            ok = (np.asarray(mask2d)[:Sq, :Skv] == 0)
            ok = ok & (j >= i - pre_tokens) & (j <= i + next_tokens)
    elif sparse_mode == 1:
        if mask2d is None:
            raise ValueError("sparse_mode 1 needs atten_mask")
        ok = (np.asarray(mask2d)[:Sq, :Skv] == 0)
    elif sparse_mode == 2:
        ok = j <= i
    elif sparse_mode == 3:
        ok = j <= i + (Skv - Sq)
    elif sparse_mode == 4:
        d = Skv - Sq
        ok = (j >= i + d - pre_tokens) & (j <= i + d + next_tokens)
    else:
        raise ValueError("sparse_mode must be 0..4")
    return np.broadcast_to(ok, (Sq, Skv)).copy()


# ---------------------------------------------------------------------------
# Step 3: softmax attention of a set of query rows over a set of key rows
#   out_i = sum_j softmax_j(scale * q_i . k_j over allowed j) v_j
#   lse_i = log(sum_j exp(s_j - max)) + max      (softmax_lse definition)
# ---------------------------------------------------------------------------
def attention_rows(Q: np.ndarray, K: np.ndarray, V: np.ndarray, allowed: np.ndarray,
                   scale: float) -> tuple[np.ndarray, np.ndarray]:
    n = Q.shape[0]
    out = np.zeros((n, V.shape[1]), dtype=np.float64)
    lse = np.full((n,), np.inf, dtype=np.float64)
    if n == 0 or K.shape[0] == 0:
        return out, lse
    s = scale * (Q @ K.T)                       # scale * Q K^T
    s = np.where(allowed, s, -np.inf)           # + atten_mask (-inf where masked)
    has = allowed.any(axis=1)
    m = np.where(has, s.max(axis=1, initial=-np.inf), 0.0)    # softmax_max
    e = np.where(allowed, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)                           # softmax_sum
    l_safe = np.where(has, l, 1.0)
    p = e / l_safe[:, None]                     # softmax
    out = np.where(has[:, None], p @ V, 0.0)
    lse = np.where(has, np.log(l_safe) + m, np.inf)
    return out, lse


# ---------------------------------------------------------------------------
# Layout views: query/key/value as [b][n] -> (S, D) row matrices
#   input_layout: BSH, BSND, BNSD, TND (npu_fused_infer_attention_score_v2).
# ---------------------------------------------------------------------------
def _as_bnsd(x: np.ndarray, layout: str, N: int) -> np.ndarray:
    if layout == "BNSD":
        return x
    if layout == "BSND":
        return x.transpose(0, 2, 1, 3)
    if layout == "BSH":
        B, S, H = x.shape
        return x.reshape(B, S, N, H // N).transpose(0, 2, 1, 3)
    raise ValueError(layout)


def _from_bnsd(x: np.ndarray, layout: str) -> np.ndarray:
    if layout == "BNSD":
        return x
    if layout == "BSND":
        return x.transpose(0, 2, 1, 3)
    if layout == "BSH":
        B, N, S, D = x.shape
        return x.transpose(0, 2, 1, 3).reshape(B, S, N * D)
    raise ValueError(layout)


def _mask_for_batch(mask, b: int):
    """atten_mask shapes (S1,S2), (B,S1,S2), (1,S1,S2), (B,1,S1,S2), (1,1,S1,S2)."""
    if mask is None:
        return None
    m = np.asarray(mask.detach().cpu().numpy() if hasattr(mask, "detach") else mask)
    if m.ndim == 2:
        return m
    if m.ndim == 3:
        return m[b if m.shape[0] > 1 else 0]
    if m.ndim == 4:
        return m[b if m.shape[0] > 1 else 0, 0]
    raise ValueError("atten_mask rank")


def fia_prefill(q, k, v, *, num_heads: int, num_key_value_heads: int = 0, scale_value: float = 1.0,
                input_layout: str = "BSH", sparse_mode: int = 0, atten_mask=None,
                actual_seq_qlen=None, actual_seq_kvlen=None,
                pre_tokens: int = INT32_MAX, next_tokens: int = INT32_MAX,
                rows=None, query_rope=None, key_rope=None):
    """Full attention (Q_S >= 1) over contiguous key/value.

    Returns (attention_out, softmax_lse) as float64 arrays: out has the query's
    shape with value's head dim; lse is (B, Q_N, Q_S, 1) or (T, Q_N, 1).
    With rows=[(b, h, i), ...] only those query rows are computed and a list of
    (out_row, lse) pairs is returned instead (used at full sizes).
    MLA prefill (npu_fused_infer_attention_score_v2, query D 128 with
    query_rope / key_rope of D 64, or query / key D 192 with value D 128): the
    score of a pair is scale * (q . k + q_rope . k_rope), i.e. the product over
    the concatenation [q, q_rope] . [k, k_rope]; value keeps its own D."""
    N1 = int(num_heads)
    N2 = int(num_key_value_heads) or N1
    if N1 % N2:
        raise ValueError("num_heads must be a multiple of num_key_value_heads")
    g = N1 // N2
    if (query_rope is None) != (key_rope is None):
        raise ValueError("query_rope and key_rope must be given together")
    Q, K, V = f64(q), f64(k), f64(v)
    if query_rope is not None:
        if input_layout == "BSH":
            # (B, S, N*D) and (B, S, N*64): concatenate per head
            B_, S1_, _ = Q.shape
            Q = np.concatenate([Q.reshape(B_, S1_, N1, -1), f64(query_rope).reshape(B_, S1_, N1, -1)],
                               axis=3).reshape(B_, S1_, -1)
            B_, S2_, _ = K.shape
            K = np.concatenate([K.reshape(B_, S2_, N2, -1), f64(key_rope).reshape(B_, S2_, N2, -1)],
                               axis=3).reshape(B_, S2_, -1)
        else:
            Q = np.concatenate([Q, f64(query_rope)], axis=-1)
            K = np.concatenate([K, f64(key_rope)], axis=-1)
    if input_layout == "TND":
        qs, ql = tnd_lengths(actual_seq_qlen)
        ks, kl = tnd_lengths(actual_seq_kvlen)
        B = len(ql)
        Dv = V.shape[2]

        def qrows(b, h): return Q[qs[b]:qs[b] + ql[b], h, :]
        def krows(b, h): return K[ks[b]:ks[b] + kl[b], h // g, :]
        def vrows(b, h): return V[ks[b]:ks[b] + kl[b], h // g, :]
    else:
        Qb, Kb, Vb = _as_bnsd(Q, input_layout, N1), _as_bnsd(K, input_layout, N2), _as_bnsd(V, input_layout, N2)
        B, Sq, Skv, Dv = Qb.shape[0], Qb.shape[2], Kb.shape[2], Vb.shape[3]
        ql = resolve_lengths(actual_seq_qlen, B, Sq)
        kl = resolve_lengths(actual_seq_kvlen, B, Skv)

        def qrows(b, h): return Qb[b, h, :ql[b], :]
        def krows(b, h): return Kb[b, h // g, :kl[b], :]
        def vrows(b, h): return Vb[b, h // g, :kl[b], :]

    def unit(b, h):
        allowed = allowed_matrix(ql[b], kl[b], sparse_mode, _mask_for_batch(atten_mask, b), pre_tokens, next_tokens)
        return allowed

    if rows is not None:
        res = []
        for (b, h, i) in rows:
            if i >= ql[b]:
                res.append((np.zeros(Dv), np.inf))
                continue
            allowed = unit(b, h)[i:i + 1]
            o, l = attention_rows(qrows(b, h)[i:i + 1], krows(b, h), vrows(b, h), allowed, scale_value)
            res.append((o[0], l[0]))
        return res

    if input_layout == "TND":
        out = np.zeros((Q.shape[0], N1, Dv))
        lse = np.full((Q.shape[0], N1, 1), np.inf)
        for b in range(B):
            for h in range(N1):
                o, l = attention_rows(qrows(b, h), krows(b, h), vrows(b, h), unit(b, h), scale_value)
                out[qs[b]:qs[b] + ql[b], h, :] = o
                lse[qs[b]:qs[b] + ql[b], h, 0] = l
        return out, lse
    out = np.zeros((B, N1, Sq, Dv))
    lse = np.full((B, N1, Sq, 1), np.inf)
    for b in range(B):
        for h in range(N1):
            o, l = attention_rows(qrows(b, h), krows(b, h), vrows(b, h), unit(b, h), scale_value)
            out[b, h, :ql[b], :] = o
            lse[b, h, :ql[b], 0] = l
    return _from_bnsd(out, input_layout), lse


# ---------------------------------------------------------------------------
# Paged KV gather (PageAttention via block_table)
#   npu_fused_infer_attention_score_v2, "page attention场景": token j of batch b
#   sits in block block_table[b][j // block_size] at row j % block_size.  The
#   cache is (blocknum, KV_N, blocksize, D) or (blocknum, blocksize, H).
# ---------------------------------------------------------------------------
def paged_rows(pool: np.ndarray, table: np.ndarray, b: int, kvh: int, L: int, bs: int, D: int) -> np.ndarray:
    rows = np.empty((L, D), dtype=np.float64)
    for j in range(L):
        blk = int(table[b, j // bs])
        r = j % bs
        if pool.ndim == 4:
            rows[j] = pool[blk, kvh, r, :]
        else:
            rows[j] = pool[blk, r, kvh * D:(kvh + 1) * D]
    return rows


def fia_decode(q, k, v, *, num_heads: int, num_key_value_heads: int = 0, scale_value: float = 1.0,
               input_layout: str = "BNSD", actual_seq_kvlen=None, block_table=None, block_size: int = 0,
               query_rope=None, key_rope=None, atten_mask=None, rows=None, sparse_mode: int = 0):
    """Incremental attention against a (paged) KV cache.  With Q_S = 1 the
    sparse_mode / pre_tokens / next_tokens parameters do not apply
    (npu_fused_infer_attention_score_v2, parameter descriptions).  With Q_S > 1
    query tokens (several new tokens per step) the mask is the formula's
    sparse_mode pattern over the Q_S x S_kv score block: 0 none, 2 left-up
    causal (j <= i), 3 right-down causal (j <= i + S_kv - Q_S, the last query
    token seeing the whole cache).

    q: BNSD (B,N1,Q_S,D), BSND (B,Q_S,N1,D) or BSH (B,Q_S,N1*D).  With
    block_table, k/v are paged pools; otherwise k/v follow input_layout.  With
    query_rope / key_rope (MLA) scores add q_rope . k_rope and key_rope is
    paged like k.  Returns (out in q's layout, lse (B, N1, Q_S, 1)); with
    rows=[(b,h)] returns pairs (out row, lse) for Q_S = 1, else (out rows
    (Q_S, D_v), lse (Q_S,))."""
    N1 = int(num_heads)
    N2 = int(num_key_value_heads) or N1
    g = N1 // N2
    Q = _as_bnsd(f64(q), input_layout, N1)
    B = Q.shape[0]
    QR = _as_bnsd(f64(query_rope), input_layout, N1) if query_rope is not None else None
    if (query_rope is None) != (key_rope is None):
        raise ValueError("query_rope and key_rope must be given together")
    Kp, Vp = f64(k), f64(v)
    KR = f64(key_rope) if key_rope is not None else None
    if block_table is not None:
        if actual_seq_kvlen is None:
            raise ValueError("page attention needs actual_seq_kvlen")
        table = np.asarray(block_table.cpu().numpy() if hasattr(block_table, "cpu") else block_table)
        kl = resolve_lengths(actual_seq_kvlen, B, table.shape[1] * block_size)
        Dk = Q.shape[3]
        Dv = Vp.shape[-1] if Vp.ndim == 4 else Vp.shape[-1] // N2
        Dr = QR.shape[3] if QR is not None else 0

        def krows(b, h):
            kk = paged_rows(Kp, table, b, h // g, kl[b], block_size, Dk)
            if KR is not None:
                kk = np.concatenate([kk, paged_rows(KR, table, b, h // g, kl[b], block_size, Dr)], axis=1)
            return kk

        def vrows(b, h): return paged_rows(Vp, table, b, h // g, kl[b], block_size, Dv)
    else:
        Kb, Vb = _as_bnsd(Kp, input_layout, N2), _as_bnsd(Vp, input_layout, N2)
        KRb = _as_bnsd(KR, input_layout, N2) if KR is not None else None
        kl = resolve_lengths(actual_seq_kvlen, B, Kb.shape[2])
        Dv = Vb.shape[3]

        def krows(b, h):
            kk = Kb[b, h // g, :kl[b], :]
            if KRb is not None:
                kk = np.concatenate([kk, KRb[b, h // g, :kl[b], :]], axis=1)
            return kk

        def vrows(b, h): return Vb[b, h // g, :kl[b], :]

    QS = Q.shape[2]

    def qrow(b, h):
        qq = Q[b, h, :, :]
        if QR is not None:
            qq = np.concatenate([qq, QR[b, h, :, :]], axis=1)
        return qq

    def allowed(b):
        m = _mask_for_batch_decode(atten_mask, b)
        ok = allowed_matrix(QS, kl[b], sparse_mode if QS > 1 else 0)
        if m is not None:
            ok = ok & (m[:kl[b]] == 0)[None, :]
        return ok

    if rows is not None:
        res = []
        cache = {}
        for (b, h) in rows:
            key = (b, h // g)
            if key not in cache:
                cache[key] = (krows(b, h), vrows(b, h))
            kk, vv = cache[key]
            o, l = attention_rows(qrow(b, h), kk, vv, allowed(b), scale_value)
            res.append((o[0], l[0]) if QS == 1 else (o, l))
        return res

    out = np.zeros((B, N1, QS, Dv))
    lse = np.full((B, N1, QS, 1), np.inf)
    for b in range(B):
        for kvh in range(N2):
            kk, vv = krows(b, kvh * g), vrows(b, kvh * g)
            for h in range(kvh * g, (kvh + 1) * g):
                o, l = attention_rows(qrow(b, h), kk, vv, allowed(b), scale_value)
                out[b, h] = o
                lse[b, h, :, 0] = l
    return _from_bnsd(out, input_layout), lse


def fia_prefill_paged(q, k, v, *, block_table, block_size: int, actual_seq_kvlen, num_heads: int,
                      num_key_value_heads: int = 0, input_layout: str = "BNSD", **prefill_kw):
    """Prefill (any Q_S) against a paged KV cache: chunked prefill, where a new
    chunk of query tokens attends to the sequence's cached keys
    (npu_fused_infer_attention_score_v2, page attention).  Key j of batch b is
    row j % block_size of block block_table[b][j // block_size] (paged_rows);
    with each batch's keys gathered that way the computation is fia_prefill's,
    under the same sparse_mode / atten_mask / pre_tokens / next_tokens.
    actual_seq_kvlen holds every batch's own key count (the cache is not TND,
    also when the query is); k / v are (blocknum, KV_N, block_size, D) or
    (blocknum, block_size, KV_N * D)."""
    N1 = int(num_heads)
    N2 = int(num_key_value_heads) or N1
    table = np.asarray(block_table.cpu().numpy() if hasattr(block_table, "cpu") else block_table)
    B = table.shape[0]
    kl = resolve_lengths(actual_seq_kvlen, B, table.shape[1] * block_size)
    Kp, Vp = f64(k), f64(v)
    Dk = Kp.shape[-1] if Kp.ndim == 4 else Kp.shape[-1] // N2
    Dv = Vp.shape[-1] if Vp.ndim == 4 else Vp.shape[-1] // N2

    def gathered(pool, D):
        per_batch = [np.stack([paged_rows(pool, table, b, h, kl[b], block_size, D) for h in range(N2)])
                     for b in range(B)]                      # (N2, L_b, D) each
        if input_layout == "TND":
            return np.concatenate([x.transpose(1, 0, 2) for x in per_batch], axis=0) if B else np.zeros((0, N2, D))
        S = max(kl) if B else 0
        out = np.zeros((B, N2, S, D))
        for b in range(B):
            out[b, :, :kl[b], :] = per_batch[b]
        return _from_bnsd(out, input_layout)

    K, V = gathered(Kp, Dk), gathered(Vp, Dv)
    kv_list = list(np.cumsum(kl)) if input_layout == "TND" else kl
    return fia_prefill(q, K, V, num_heads=N1, num_key_value_heads=N2, input_layout=input_layout,
                       actual_seq_kvlen=kv_list, **prefill_kw)


def _mask_for_batch_decode(mask, b: int):
    """Decode atten_mask shapes (B, KV_S), (B, 1, KV_S), (B, 1, 1, KV_S)."""
    if mask is None:
        return None
    m = np.asarray(mask.detach().cpu().numpy() if hasattr(mask, "detach") else mask)
    return m.reshape(m.shape[0], -1)[b if m.shape[0] > 1 else 0]


# ---------------------------------------------------------------------------
# Block-sparse attention (aclnnBlockSparseAttentionV2)
#   attentionOut = Softmax(scale * query * key_sparse^T) * value_sparse, where
#   the keys of query row i are those in the KV blocks that
#   blockSparseMask[b, h, i // X, j // Y] selects; blocks are X x Y with
#   ceil division, so the last row/column block may be partial.
# ---------------------------------------------------------------------------
def bsa_forward(q, k, v, block_sparse_mask, block_shape, *, num_heads: int, num_key_value_heads: int = 0,
                scale_value: float = 1.0, input_layout: str = "BNSD",
                actual_seq_qlen=None, actual_seq_kvlen=None, rows=None,
                q_dequant_scale=None, k_dequant_scale=None, v_dequant_scale=None):
    """Block-sparse attention (aclnnBlockSparseAttentionV2, "计算公式").

    FP8 inputs ("FP8特性说明"): q / k / v hold float8_e4m3fn values and the
    dequant scales say what each block of rows is worth: row i of query head h
    of batch b is q[i] * q_dequant_scale[b, h, i // X, 0], key / value row j
    of kv head n is k[j] * k_dequant_scale[b, n, j // Y, 0] (and v with
    v_dequant_scale), X / Y = block_shape (the pages tie the quantisation
    blocks to block_shape: 128 query rows, 256 or 512 key rows).  Attention
    then runs on the dequantised values."""
    X, Y = int(block_shape[0]), int(block_shape[1])
    M = np.asarray(block_sparse_mask.cpu().numpy() if hasattr(block_sparse_mask, "cpu") else block_sparse_mask)
    N1 = int(num_heads)
    N2 = int(num_key_value_heads) or N1
    g = N1 // N2
    Q, K, V = f64(q), f64(k), f64(v)
    scales = (q_dequant_scale, k_dequant_scale, v_dequant_scale)
    if any(x is not None for x in scales) and any(x is None for x in scales):
        raise ValueError("FP8 needs all three dequant scales")
    fp8 = q_dequant_scale is not None
    if fp8:
        QSC, KSC, VSC = (f64(x)[..., 0] for x in scales)   # (B, heads, blocks)
    if input_layout == "TND":
        qs, ql = tnd_lengths(actual_seq_qlen)
        ks, kl = tnd_lengths(actual_seq_kvlen)
        B = len(ql)
        if fp8:
            # step 0: dequantise every row by its block's scale
            for b in range(B):
                iq, jk = np.arange(ql[b]) // X, np.arange(kl[b]) // Y
                Q[qs[b]:qs[b] + ql[b]] *= QSC[b][:, iq].T[:, :, None]
                K[ks[b]:ks[b] + kl[b]] *= KSC[b][:, jk].T[:, :, None]
                V[ks[b]:ks[b] + kl[b]] *= VSC[b][:, jk].T[:, :, None]

        def qrows(b, h): return Q[qs[b]:qs[b] + ql[b], h, :]
        def krows(b, h): return K[ks[b]:ks[b] + kl[b], h // g, :]
        def vrows(b, h): return V[ks[b]:ks[b] + kl[b], h // g, :]
    else:
        Qb, Kb, Vb = _as_bnsd(Q, input_layout, N1), _as_bnsd(K, input_layout, N2), _as_bnsd(V, input_layout, N2)
        B = Qb.shape[0]
        ql = resolve_lengths(actual_seq_qlen, B, Qb.shape[2])
        kl = resolve_lengths(actual_seq_kvlen, B, Kb.shape[2])
        if fp8:
            # step 0: dequantise every row by its block's scale (views of Q / K / V)
            for b in range(B):
                iq, jk = np.arange(ql[b]) // X, np.arange(kl[b]) // Y
                Qb[b, :, :ql[b]] *= QSC[b][:, iq][:, :, None]
                Kb[b, :, :kl[b]] *= KSC[b][:, jk][:, :, None]
                Vb[b, :, :kl[b]] *= VSC[b][:, jk][:, :, None]

        def qrows(b, h): return Qb[b, h, :ql[b], :]
        def krows(b, h): return Kb[b, h // g, :kl[b], :]
        def vrows(b, h): return Vb[b, h // g, :kl[b], :]

    def allowed(b, h, i0, i1):
        i = np.arange(i0, i1)[:, None]
        j = np.arange(kl[b])[None, :]
        return M[b, h][i // X, j // Y] != 0

    if rows is not None:
        res = []
        for (b, h, i) in rows:
            if i >= ql[b]:
                res.append((np.zeros(V.shape[-1]), np.inf))
                continue
            o, l = attention_rows(qrows(b, h)[i:i + 1], krows(b, h), vrows(b, h), allowed(b, h, i, i + 1), scale_value)
            res.append((o[0], l[0]))
        return res

    Dv = V.shape[-1]
    if input_layout == "TND":
        out = np.zeros((Q.shape[0], N1, Dv))
        lse = np.full((Q.shape[0], N1, 1), np.inf)
    else:
        out = np.zeros((B, N1, Qb.shape[2], Dv))
        lse = np.full((B, N1, Qb.shape[2], 1), np.inf)
    for b in range(B):
        for h in range(N1):
            o, l = attention_rows(qrows(b, h), krows(b, h), vrows(b, h), allowed(b, h, 0, ql[b]), scale_value)
            if input_layout == "TND":
                out[qs[b]:qs[b] + ql[b], h] = o
                lse[qs[b]:qs[b] + ql[b], h, 0] = l
            else:
                out[b, h, :ql[b]] = o
                lse[b, h, :ql[b], 0] = l
    if input_layout == "TND":
        return out, lse
    return _from_bnsd(out, input_layout), lse


# ---------------------------------------------------------------------------
# Merging partial results over disjoint key sets by their LSE
#   npu_fused_infer_attention_score_v2, return_softmax_lse: the LSE output exists
#   so that attention split along the key axis (ring attention) can be merged.
#   A part with no keys (lse = +inf by the empty rule) contributes nothing.
# ---------------------------------------------------------------------------
def lse_merge(outs, lses):
    outs = [np.asarray(o, dtype=np.float64) for o in outs]
    lses = [np.asarray(l, dtype=np.float64) for l in lses]
    live = [np.isfinite(l) for l in lses]
    m = np.full(lses[0].shape, -np.inf)
    for l, ok in zip(lses, live):
        m = np.where(ok, np.maximum(m, l), m)
    any_live = np.isfinite(m)
    m0 = np.where(any_live, m, 0.0)
    total = np.zeros(lses[0].shape)
    for l, ok in zip(lses, live):
        total += np.where(ok, np.exp(np.where(ok, l, 0.0) - m0), 0.0)
    lse = np.where(any_live, np.log(np.where(any_live, total, 1.0)) + m0, np.inf)
    out = np.zeros(outs[0].shape)
    for o, l, ok in zip(outs, lses, live):
        w = np.where(ok & any_live, np.exp(np.where(ok, l, 0.0) - np.where(any_live, lse, 0.0)), 0.0)
        out += w[..., None] * o
    return out, lse

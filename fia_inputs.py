"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the CPU oracle.

This module only draws random numbers and arranges them into tensors of the
shapes the FusedInferAttentionScore / PromptFlashAttention / BlockSparseAttention
pages describe.  It holds none of the attention arithmetic.

Every tensor comes from numpy's PCG64 seeded with (BASE_SEED, workload id,
tensor id), is drawn in float32 and cast to fp16/bf16 with round-to-nearest-even
by torch.  All tensors are returned on the CPU; callers move them where needed.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BASE_SEED = 20261202

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16, "f32": torch.float32}


def rng(workload: int, tensor: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([BASE_SEED, workload, tensor])))


def normal(shape, dtype: str, workload: int, tensor: int) -> torch.Tensor:
    x = rng(workload, tensor).standard_normal(size=tuple(shape), dtype=np.float32)
    return torch.from_numpy(x).to(DTYPES[dtype])


def uniform_ints(lo: int, hi: int, n: int, workload: int, tensor: int) -> list[int]:
    """n integers uniform on [lo, hi] (inclusive)."""
    return [int(v) for v in rng(workload, tensor).integers(lo, hi + 1, size=n)]


def cumsum_no_leading_zero(lengths):
    out, acc = [], 0
    for n in lengths:
        acc += int(n)
        out.append(acc)
    return out


# --------------------------------------------------------------------------------------
# Dense prefill (BNSD / BSND / BSH / TND)
# --------------------------------------------------------------------------------------
@dataclass
class PrefillCase:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    num_heads: int
    num_key_value_heads: int
    scale: float
    layout: str
    sparse_mode: int
    actual_seq_qlen: list | None = None
    actual_seq_kvlen: list | None = None
    atten_mask: torch.Tensor | None = None
    lse: bool = True
    meta: dict = field(default_factory=dict)


def prefill_case(B, N1, N2, Sq, Skv, D, dtype="bf16", layout="BNSD", sparse_mode=0,
                 actual_seq_qlen=None, actual_seq_kvlen=None, workload=100, Dv=None,
                 poison_padding=False) -> PrefillCase:
    """Dense q/k/v with iid N(0,1) entries in the given layout.

    With poison_padding, key/value rows past each batch's actual kv length are
    set to NaN: a correct implementation never lets them reach the output."""
    Dv = D if Dv is None else Dv
    if layout == "BNSD":
        qs, ks, vs = (B, N1, Sq, D), (B, N2, Skv, D), (B, N2, Skv, Dv)
    elif layout == "BSND":
        qs, ks, vs = (B, Sq, N1, D), (B, Skv, N2, D), (B, Skv, N2, Dv)
    elif layout == "BSH":
        qs, ks, vs = (B, Sq, N1 * D), (B, Skv, N2 * D), (B, Skv, N2 * Dv)
    else:
        raise ValueError(layout)
    q = normal(qs, dtype, workload, 1)
    k = normal(ks, dtype, workload, 2)
    v = normal(vs, dtype, workload, 3)
    if poison_padding and actual_seq_kvlen is not None:
        for b in range(B):
            L = actual_seq_kvlen[0] if len(actual_seq_kvlen) == 1 else actual_seq_kvlen[b]
            if layout == "BNSD":
                k[b, :, L:] = float("nan"); v[b, :, L:] = float("nan")
            else:
                k[b, L:] = float("nan"); v[b, L:] = float("nan")
    return PrefillCase(q, k, v, N1, N2, 1.0 / math.sqrt(D), layout, sparse_mode,
                       actual_seq_qlen, actual_seq_kvlen)


def tnd_case(lengths_q, lengths_kv, N1, N2, D, dtype="bf16", sparse_mode=3, workload=300) -> PrefillCase:
    Tq, Tkv = sum(lengths_q), sum(lengths_kv)
    q = normal((Tq, N1, D), dtype, workload, 1)
    k = normal((Tkv, N2, D), dtype, workload, 2)
    v = normal((Tkv, N2, D), dtype, workload, 3)
    return PrefillCase(q, k, v, N1, N2, 1.0 / math.sqrt(D), "TND", sparse_mode,
                       cumsum_no_leading_zero(lengths_q), cumsum_no_leading_zero(lengths_kv))


def atten_mask(shape, kind="random", density=0.3, dtype="u8", workload=600) -> torch.Tensor:
    """Seeded atten_mask of the given shape (..., S1m, S2m); nonzero = masked.

    kind "random": i.i.d. entries, `density` of them nonzero.  "blocks": each
    128 x 128 tile is all visible, all masked or random (a third each), and a
    few rows are masked in full.  "causal": key j of row i masked when j > i.
    Nonzero entries take assorted values (1..255 for uint8, nonzero int8)."""
    g = rng(workload, 50)
    S1, S2 = shape[-2], shape[-1]
    if kind == "causal":
        m = np.broadcast_to(np.arange(S2)[None, :] > np.arange(S1)[:, None], shape)
    elif kind == "random":
        m = g.random(size=shape) < density
    elif kind == "blocks":
        m = g.random(size=shape) < density
        t1, t2 = -(-S1 // 128), -(-S2 // 128)
        pick = g.integers(0, 3, size=tuple(shape[:-2]) + (t1, t2))
        full = np.repeat(np.repeat(pick, 128, axis=-2), 128, axis=-1)[..., :S1, :S2]
        m = np.where(full == 0, False, np.where(full == 1, True, m))
        rows = g.integers(0, S1, size=max(1, S1 // 64))
        m[..., rows, :] = True
    else:
        raise ValueError(kind)
    m = np.ascontiguousarray(m)
    if dtype == "bool":
        return torch.from_numpy(m.copy())
    if dtype == "u8":
        vals = g.integers(1, 256, size=m.shape)
    else:
        vals = g.choice(np.r_[np.arange(-128, 0), np.arange(1, 128)], size=m.shape)
    out = np.where(m, vals, 0).astype(np.uint8 if dtype == "u8" else np.int8)
    return torch.from_numpy(out)


# The five workloads the pages' operator is exercised on (sizes fixed here).
def workload_prefill_bnsd_f16_small() -> PrefillCase:
    """Prefill BNSD fp16: B=1, Q_N=KV_N=2, S=128, D=64, causal, LSE on."""
    return prefill_case(1, 2, 2, 128, 128, 64, dtype="f16", layout="BNSD", sparse_mode=2, workload=1)


def workload_tnd_varlen(n_seq=8, lo=256, hi=4096, N1=32, N2=8, D=128, workload=3) -> PrefillCase:
    """Varlen TND bf16 prefill: n_seq lengths uniform on [lo, hi], causal, GQA 32/8."""
    lens = uniform_ints(lo, hi, n_seq, workload, 0)
    return tnd_case(lens, lens, N1, N2, D, "bf16", sparse_mode=3, workload=workload)


# --------------------------------------------------------------------------------------
# Paged decode
# --------------------------------------------------------------------------------------
@dataclass
class DecodeCase:
    q: torch.Tensor               # BNSD (B, N1, 1, D)
    k_pool: torch.Tensor          # (nblk, N2, bs, D)
    v_pool: torch.Tensor
    block_table: torch.Tensor     # int32 (B, max_blocks)
    kv_lens: list
    block_size: int
    num_heads: int
    num_key_value_heads: int
    scale: float
    meta: dict = field(default_factory=dict)


def paged_decode_case(B, N1, N2, D, kv_lens, block_size=128, dtype="bf16", workload=200,
                      extra_table_cols=1, poison=True, layout_kv="BNBD", q_tokens=1) -> DecodeCase:
    """Paged KV cache: each sequence's logical blocks map to a random permutation of
    a shared physical pool.  One extra pool block is filled with NaN; unused
    block_table entries point at it, as do the unused tail rows of each sequence's
    last block, so any read past a sequence's length poisons the output."""
    nb = [(L + block_size - 1) // block_size for L in kv_lens]
    total = sum(nb)
    nblk = total + 1
    poison_id = total
    perm = rng(workload, 10).permutation(total)
    max_blocks = max(max(nb), 1) + extra_table_cols
    table = np.full((B, max_blocks), poison_id, dtype=np.int32)
    pos = 0
    for b in range(B):
        for i in range(nb[b]):
            table[b, i] = perm[pos]
            pos += 1
    if layout_kv == "BNBD":
        shape = (nblk, N2, block_size, D)
    else:  # (blocknum, blocksize, H)
        shape = (nblk, block_size, N2 * D)
    k = normal(shape, dtype, workload, 2)
    v = normal(shape, dtype, workload, 3)
    if poison:
        k[poison_id] = float("nan")
        v[poison_id] = float("nan")
        for b in range(B):
            tail = kv_lens[b] % block_size
            if nb[b] and tail:
                last = int(table[b, nb[b] - 1])
                if layout_kv == "BNBD":
                    k[last, :, tail:] = float("nan"); v[last, :, tail:] = float("nan")
                else:
                    k[last, tail:] = float("nan"); v[last, tail:] = float("nan")
    q = normal((B, N1, q_tokens, D), dtype, workload, 1)
    return DecodeCase(q, k, v, torch.from_numpy(table), list(kv_lens), block_size, N1, N2,
                      1.0 / math.sqrt(D), {"poison_block": poison_id, "layout_kv": layout_kv})


def workload_paged_gqa_decode(B=16, N1=32, N2=8, D=128, max_len=4096, workload=2) -> DecodeCase:
    """Decode GQA bf16 with paged KV: lengths uniform on [1, max_len], block 128."""
    lens = uniform_ints(1, max_len, B, workload, 0)
    return paged_decode_case(B, N1, N2, D, lens, 128, "bf16", workload)


# --------------------------------------------------------------------------------------
# MLA prefill (scores over 192 columns, value 128)
# --------------------------------------------------------------------------------------
@dataclass
class MLAPrefillCase:
    q: torch.Tensor                   # (.., 192), or (.., 128) with q_rope (.., 64)
    k: torch.Tensor
    v: torch.Tensor                   # (.., 128)
    q_rope: torch.Tensor | None
    k_rope: torch.Tensor | None
    num_heads: int
    num_key_value_heads: int
    scale: float
    layout: str
    actual_seq_qlen: list | None = None
    actual_seq_kvlen: list | None = None


def mla_prefill_case(lens_q, lens_kv, N1, N2, rope=True, dtype="bf16", layout="TND", workload=800) -> MLAPrefillCase:
    """MLA prefill inputs: with rope, q/k of D 128 plus q_rope/k_rope of D 64,
    else q/k of D 192; v of D 128; scale 1/sqrt(192).  TND takes cumulative
    lists; the padded layouts take B = len(lens_q) and S = max length."""
    dq = 128 if rope else 192

    def shaped(n_heads, d, lens, tensor):
        if layout == "TND":
            return normal((sum(lens), n_heads, d), dtype, workload, tensor)
        B, S = len(lens), max(lens) if lens else 0
        shape = {"BNSD": (B, n_heads, S, d), "BSND": (B, S, n_heads, d), "BSH": (B, S, n_heads * d)}[layout]
        return normal(shape, dtype, workload, tensor)

    q, k, v = shaped(N1, dq, lens_q, 1), shaped(N2, dq, lens_kv, 2), shaped(N2, 128, lens_kv, 3)
    qr = shaped(N1, 64, lens_q, 4) if rope else None
    kr = shaped(N2, 64, lens_kv, 5) if rope else None
    if layout == "TND":
        aq, ak = cumsum_no_leading_zero(lens_q), cumsum_no_leading_zero(lens_kv)
    else:
        aq, ak = list(lens_q), list(lens_kv)
    return MLAPrefillCase(q, k, v, qr, kr, N1, N2, 1.0 / math.sqrt(192), layout, aq, ak)


def workload_mla_prefill(n_seq=8, lo=256, hi=4096, N=32, workload=3) -> MLAPrefillCase:
    """MLA prefill bf16, TND: the varlen prefill lengths, 32 heads (MHA), query
    and key D 192 (128 + 64 rope columns), value D 128, causal."""
    lens = uniform_ints(lo, hi, n_seq, workload, 0)
    return mla_prefill_case(lens, lens, N, N, rope=False, dtype="bf16", layout="TND", workload=810)


# --------------------------------------------------------------------------------------
# Prefill against a paged cache (chunked prefill)
# --------------------------------------------------------------------------------------
@dataclass
class PagedPrefillCase:
    q: torch.Tensor               # BNSD (B, N1, max q_len, D) / BSND / BSH, or TND (T, N1, D)
    k_pool: torch.Tensor          # (nblk, N2, bs, D) or (nblk, bs, N2*D)
    v_pool: torch.Tensor
    block_table: torch.Tensor     # int32 (B, max_blocks)
    q_lens: list
    kv_lens: list
    actual_seq_qlen: list         # per batch, or cumulative for TND
    block_size: int
    num_heads: int
    num_key_value_heads: int
    scale: float
    layout: str
    meta: dict = field(default_factory=dict)


def paged_prefill_case(q_lens, kv_lens, N1, N2, D, block_size=256, dtype="bf16", layout="BNSD", layout_kv="BNBD",
                       workload=700) -> PagedPrefillCase:
    """A chunk of q_lens[b] new query rows per sequence against kv_lens[b]
    cached keys (the chunk's own keys included) in a paged pool built like
    paged_decode_case's: shuffled blocks, a NaN block behind unused table
    entries, NaN rows past each sequence's length in its last block."""
    B = len(kv_lens)
    dc = paged_decode_case(B, N1, N2, D, kv_lens, block_size, dtype, workload, layout_kv=layout_kv)
    if layout == "TND":
        q = normal((sum(q_lens), N1, D), dtype, workload, 20)
        aq = cumsum_no_leading_zero(q_lens)
    else:
        S = max(q_lens) if q_lens else 0
        shape = {"BNSD": (B, N1, S, D), "BSND": (B, S, N1, D), "BSH": (B, S, N1 * D)}[layout]
        q = normal(shape, dtype, workload, 20)
        aq = list(q_lens)
    return PagedPrefillCase(q, dc.k_pool, dc.v_pool, dc.block_table, list(q_lens), list(kv_lens), aq, block_size,
                            N1, N2, 1.0 / math.sqrt(D), layout, {"layout_kv": layout_kv, **dc.meta})


def workload_chunked_prefill(B=8, chunk=2048, max_ctx=14336, N1=32, N2=8, D=128, block_size=256,
                             workload=6) -> PagedPrefillCase:
    """Chunked prefill bf16: a 2048-token chunk per sequence after a cached
    context uniform on [0, max_ctx], paged in 256-token blocks, GQA 32/8."""
    ctx = uniform_ints(0, max_ctx, B, workload, 0)
    return paged_prefill_case([chunk] * B, [c + chunk for c in ctx], N1, N2, D, block_size, "bf16", "BNSD", "BNBD",
                              workload)


# --------------------------------------------------------------------------------------
# MLA decode
# --------------------------------------------------------------------------------------
@dataclass
class MLACase:
    q: torch.Tensor            # BSND (B, 1, N1, 512)
    q_rope: torch.Tensor       # (B, 1, N1, 64)
    latent: torch.Tensor       # (nblk, bs, 512)  -- key and value
    rope: torch.Tensor         # (nblk, bs, 64)
    block_table: torch.Tensor  # int32 (B, max_blocks)
    kv_lens: list
    block_size: int
    num_heads: int
    scale: float


def mla_decode_case(B, N1, kv_lens, block_size=128, Dl=512, Dr=64, workload=400, extra_blocks=0,
                    poison=False) -> MLACase:
    """Paged latent + rope caches.  With poison=True one extra block is NaN and
    unused block_table entries point at it, and the rows past each sequence's
    length in its last block are NaN, so a read outside a sequence is seen."""
    nb = [(L + block_size - 1) // block_size for L in kv_lens]
    total = sum(nb) + extra_blocks
    perm = rng(workload, 10).permutation(total)
    max_blocks = max(max(nb), 1)
    nblk = total + (1 if poison else 0)
    unused = total if poison else (perm[-1] if total else 0)
    table = np.zeros((B, max_blocks), dtype=np.int32)
    pos = 0
    for b in range(B):
        for i in range(max_blocks):
            if i < nb[b]:
                table[b, i] = perm[pos]; pos += 1
            else:
                table[b, i] = unused
    latent = normal((nblk, block_size, Dl), "bf16", workload, 2)
    rope = normal((nblk, block_size, Dr), "bf16", workload, 3)
    if poison:
        latent[total] = float("nan"); rope[total] = float("nan")
        for b in range(B):
            tail = kv_lens[b] % block_size
            if nb[b] and tail:
                last = int(table[b, nb[b] - 1])
                latent[last, tail:] = float("nan"); rope[last, tail:] = float("nan")
    q = normal((B, 1, N1, Dl), "bf16", workload, 1)
    qr = normal((B, 1, N1, Dr), "bf16", workload, 4)
    return MLACase(q, qr, latent, rope, torch.from_numpy(table), list(kv_lens), block_size, N1,
                   1.0 / math.sqrt(Dl + Dr))


def workload_mla_decode(B=32, N1=128, L=8192, workload=4) -> MLACase:
    """MLA decode bf16: 128 heads, 512-d latent + 64-d rope, kv length L, block 128."""
    return mla_decode_case(B, N1, [L] * B, 128, workload=workload)


# --------------------------------------------------------------------------------------
# Block-sparse prefill
# --------------------------------------------------------------------------------------
@dataclass
class BSACase:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    mask: torch.Tensor         # uint8 (B, N1, ceil(Sq/X), ceil(Skv/Y)), nonzero = keep
    block_shape: tuple
    num_heads: int
    num_key_value_heads: int
    scale: float
    layout: str
    actual_seq_qlen: list | None = None
    actual_seq_kvlen: list | None = None


def bsa_case(B, N1, N2, Sq, Skv, D, X=128, Y=128, keep=0.25, dtype="bf16", workload=500,
             diagonal=True) -> BSACase:
    """BNSD q/k/v and a block mask keeping the diagonal block plus each other
    block with probability `keep` (seeded Bernoulli)."""
    q = normal((B, N1, Sq, D), dtype, workload, 1)
    k = normal((B, N2, Skv, D), dtype, workload, 2)
    v = normal((B, N2, Skv, D), dtype, workload, 3)
    nq, nk = -(-Sq // X), -(-Skv // Y)
    u = rng(workload, 5).random(size=(B, N1, nq, nk))
    m = (u < keep).astype(np.uint8)
    if diagonal:
        for i in range(nq):
            # the KV block holding the same token positions as query block i
            j = min((i * X) // Y, nk - 1)
            m[:, :, i, j] = 1
    return BSACase(q, k, v, torch.from_numpy(m), (X, Y), N1, N2, 1.0 / math.sqrt(D), "BNSD")


@dataclass
class BSAFp8Case:
    base: BSACase              # q / k / v float8 e4m3, the block mask, block_shape (128, Y)
    q_scale: torch.Tensor      # fp32 (B, N1, ceil(Sq/128), 1)
    k_scale: torch.Tensor      # fp32 (B, N2, ceil(Skv/Y), 1)
    v_scale: torch.Tensor


def fp8_e4m3(shape, workload: int, tensor: int, spread: float = 16.0) -> torch.Tensor:
    """float8 e4m3 values: N(0,1) * spread, clipped to the format's +-448 and
    rounded to nearest by torch."""
    x = rng(workload, tensor).standard_normal(size=tuple(shape), dtype=np.float32) * spread
    return torch.from_numpy(np.clip(x, -448.0, 448.0)).to(torch.float8_e4m3fn)


def bsa_fp8_case(B, N1, N2, Sq, Skv, Y=256, keep=0.25, workload=600, layout="BNSD") -> BSAFp8Case:
    """FP8 block-sparse inputs (D = 128): e4m3 q / k / v of spread 16, dequant
    scales uniform on [0.5, 1.5] / 16 per block of 128 query rows / Y key rows,
    the block mask of bsa_case (128 x Y blocks: diagonal + Bernoulli(keep))."""
    c = bsa_case(B, N1, N2, Sq, Skv, 128, 128, Y, keep, "bf16", workload)
    c.q, c.k, c.v = (fp8_e4m3(t.shape, workload, 20 + n) for n, t in enumerate((c.q, c.k, c.v)))
    nq, nk = -(-Sq // 128), -(-Skv // Y)
    g = rng(workload, 30)
    qs = torch.from_numpy((g.random((B, N1, nq, 1)) + 0.5).astype(np.float32) / 16)
    ks = torch.from_numpy((g.random((B, N2, nk, 1)) + 0.5).astype(np.float32) / 16)
    vs = torch.from_numpy((g.random((B, N2, nk, 1)) + 0.5).astype(np.float32) / 16)
    if layout == "BSND":
        c.q, c.k, c.v = (t.transpose(1, 2).contiguous() for t in (c.q, c.k, c.v))
        c.layout = "BSND"
    return BSAFp8Case(c, qs, ks, vs)


def workload_bsa(B=2, N1=32, N2=8, S=16384, D=128, workload=5) -> BSACase:
    """Block-sparse prefill bf16: 128x128 blocks, diagonal + ~25% of the rest."""
    return bsa_case(B, N1, N2, S, S, D, 128, 128, 0.25, "bf16", workload)


def workload_fp8_dense(B=2, N1=32, N2=8, S=4096, workload=6) -> BSAFp8Case:
    """Dense FP8 e4m3 prefill (D = 128, no mask: every key): B=2, 32/8 heads,
    S=4096, per-block dequant scales of 128 query rows / 256 key rows.  The
    case's block mask is all ones (what the oracle and the FLOP count take);
    the call passes none."""
    f = bsa_fp8_case(B, N1, N2, S, S, 256, 1.0, workload)
    f.base.mask = torch.ones_like(f.base.mask)
    return f


def workload_bsa_fp8(B=2, N1=32, N2=8, S=16384, workload=5) -> BSAFp8Case:
    """Block-sparse prefill FP8 e4m3 (D = 128): 128 x 256 blocks (the
    quantisation blocks), diagonal + ~25% of the rest."""
    return bsa_fp8_case(B, N1, N2, S, S, 256, 0.25, workload)

"""The oracle against its pins (CPU only), and proof that the pins bite:
plausible mistakes planted in copies of the oracle each fail at least one pin."""
import math
import types

import numpy as np
import pytest

from oracle import fia_oracle
from tests import pins
from tests.golden.fixtures import read_kv, shape
import fia_inputs


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda c: c.__name__)
def test_pin(check):
    check(fia_oracle)


# (old text, new text, what the mistake is)
MUTATIONS = [
    ("s = scale * (Q @ K.T)", "s = (Q @ K.T)", "dropped scale"),
    ("lse = np.where(has, np.log(l_safe) + m, np.inf)", "lse = np.where(has, np.log(l_safe), np.inf)",
     "lse without the max"),
    ("def krows(b, h): return Kb[b, h // g, :kl[b], :]", "def krows(b, h): return Kb[b, h % N2, :kl[b], :]",
     "GQA heads interleaved"),
    ("ok = j <= i + (Skv - Sq)", "ok = j <= i", "mode 3 anchored top-left"),
    ("ok = j <= i\n", "ok = j < i\n", "mode 2 excludes the diagonal"),
    ("ok = (np.asarray(mask2d)[:Sq, :Skv] == 0)\n    elif", "ok = (np.asarray(mask2d)[:Sq, :Skv] != 0)\n    elif",
     "mask polarity"),
    ("blk = int(table[b, j // bs])\n        r = j % bs", "blk = int(table[b, j % bs])\n        r = j // bs",
     "paged index swapped"),
    ("starts.append(prev)\n        lens.append(c - prev)", "starts.append(prev)\n        lens.append(c)",
     "TND list read as lengths"),
    ("return M[b, h][i // X, j // Y] != 0", "return M[b, h][i // Y, j // X] != 0", "BSA block shape swapped"),
    ("p = e / l_safe[:, None]", "p = e", "missing normalisation"),
    ("w = np.where(ok & any_live, np.exp(np.where(ok, l, 0.0) - np.where(any_live, lse, 0.0)), 0.0)",
     "w = np.where(ok & any_live, 1.0, 0.0)", "merge without weights"),
    ("kl = resolve_lengths(actual_seq_kvlen, B, Kb.shape[2])\n        Dv = Vb.shape[3]",
     "kl = resolve_lengths(None, B, Kb.shape[2])\n        Dv = Vb.shape[3]", "decode ignores kv lengths"),
    ("kk = np.concatenate([kk, paged_rows(KR, table, b, h // g, kl[b], block_size, Dr)], axis=1)",
     "kk = kk", "MLA rope term dropped"),
    ("ok = allowed_matrix(QS, kl[b], sparse_mode if QS > 1 else 0)", "ok = allowed_matrix(QS, kl[b], 0)",
     "multi-token decode ignores its mask"),
    ("qq = Q[b, h, :, :]", "qq = Q[b, h, :1, :]", "multi-token decode uses the first token only"),
    ("per_batch = [np.stack([paged_rows(pool, table, b, h, kl[b], block_size, D) for h in range(N2)])",
     "per_batch = [np.stack([paged_rows(pool, table, b, 0, kl[b], block_size, D) for h in range(N2)])",
     "paged prefill reads kv head 0 only"),
    ("kv_list = list(np.cumsum(kl)) if input_layout == \"TND\" else kl", "kv_list = kl",
     "paged prefill TND kv list not cumulative"),
    ("            K = np.concatenate([K, f64(key_rope)], axis=-1)",
     "            K = np.concatenate([K, 0 * f64(key_rope)], axis=-1)", "MLA prefill rope term dropped"),
    ("            Q = np.concatenate([Q, f64(query_rope)], axis=-1)",
     "            Q = np.concatenate([f64(query_rope), Q], axis=-1)", "MLA prefill rope on the wrong side"),
    ("                iq, jk = np.arange(ql[b]) // X, np.arange(kl[b]) // Y\n                Qb[",
     "                iq, jk = np.arange(ql[b]) // Y, np.arange(kl[b]) // Y\n                Qb[",
     "FP8 query blocks sized like key blocks"),
    ("                Vb[b, :, :kl[b]] *= VSC[b][:, jk][:, :, None]", "                pass",
     "FP8 value scales dropped"),
    ("                K[ks[b]:ks[b] + kl[b]] *= KSC[b][:, jk].T[:, :, None]", "                pass",
     "FP8 TND key scales dropped"),
    ("        return m[b if m.shape[0] > 1 else 0]\n", "        return m[0]\n", "3-D atten_mask reads batch 0"),
    ("        return m[b if m.shape[0] > 1 else 0, 0]", "        return m[0, 0]", "4-D atten_mask reads batch 0"),
    ("    return m.reshape(m.shape[0], -1)[b if m.shape[0] > 1 else 0]", "    return m.reshape(m.shape[0], -1)[0]",
     "decode atten_mask reads batch 0"),
    ("            ok = ok & (m[:kl[b]] == 0)[None, :]", "            ok = ok & (m[:kl[b]] != 0)[None, :]",
     "decode atten_mask polarity"),
]


def _mutant(old, new):
    import inspect
    src = inspect.getsource(fia_oracle)
    assert old in src, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("fia_oracle_mutant")
    exec(compile(src.replace(old, new, 1), "fia_oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("old,new,what", MUTATIONS, ids=[m[2] for m in MUTATIONS])
def test_pins_catch_planted_mistake(old, new, what):
    mod = _mutant(old, new)
    failed = []
    for check in pins.ALL_CHECKS:
        try:
            check(mod)
        except Exception:
            failed.append(check.__name__)
    assert failed, f"no pin caught: {what}"


def test_worked_example_shape():
    """npu_prompt_flash_attention call example: q (1,8,164,128) fp16 against
    k/v (1,8,1024,128) gives out (1,8,164,128) fp16 (values not reproducible)."""
    fx = read_kv("pfa_worked_example.txt")
    B, N, Sq, D = shape(fx["q_shape"])
    Skv = shape(fx["k_shape"])[2]
    case = fia_inputs.prefill_case(B, N, N, Sq, Skv, D, dtype="f16", layout="BNSD", workload=7)
    rows = [(0, h, i) for h in (0, 7) for i in (0, 163)]
    res = fia_oracle.fia_prefill(case.q, case.k, case.v, num_heads=int(fx["num_heads"]),
                                 scale_value=float(fx["scale_value"]), input_layout=fx["input_layout"],
                                 actual_seq_qlen=[int(fx["actual_seq_lengths"])],
                                 actual_seq_kvlen=[int(fx["actual_seq_lengths_kv"])],
                                 pre_tokens=int(fx["pre_tokens"]), next_tokens=int(fx["next_tokens"]), rows=rows)
    assert all(o.shape == (D,) and np.isfinite(l) for o, l in res)
    out, lse = fia_oracle.fia_prefill(case.q[:, :1, :3], case.k[:, :1], case.v[:, :1], num_heads=1,
                                      scale_value=float(fx["scale_value"]), input_layout="BNSD")
    assert out.shape == (1, 1, 3, D)
    assert shape(fx["out_shape"]) == (B, N, Sq, D)
    assert abs(float(fx["scale_value"]) - 1 / math.sqrt(128)) < 1e-15


def test_sampled_rows_match_full():
    case = fia_inputs.tnd_case([5, 9], [5, 9], 4, 2, 8, workload=9)
    out, lse = fia_oracle.fia_prefill(case.q, case.k, case.v, num_heads=4, num_key_value_heads=2,
                                      scale_value=case.scale, input_layout="TND", sparse_mode=3,
                                      actual_seq_qlen=case.actual_seq_qlen, actual_seq_kvlen=case.actual_seq_kvlen)
    rows = [(0, 1, 4), (1, 3, 0), (1, 0, 8)]
    res = fia_oracle.fia_prefill(case.q, case.k, case.v, num_heads=4, num_key_value_heads=2,
                                 scale_value=case.scale, input_layout="TND", sparse_mode=3,
                                 actual_seq_qlen=case.actual_seq_qlen, actual_seq_kvlen=case.actual_seq_kvlen,
                                 rows=rows)
    starts = [0, 5]
    for (b, h, i), (o, l) in zip(rows, res):
        assert np.allclose(o, out[starts[b] + i, h]) and np.isclose(l, lse[starts[b] + i, h, 0])


def test_resolve_lengths_rules():
    """actual_seq_* list rules: length 1 broadcasts, >= B takes the first B,
    anything else (or an entry above S) is an error."""
    assert fia_oracle.resolve_lengths([3], 4, 5) == [3, 3, 3, 3]
    assert fia_oracle.resolve_lengths([1, 2, 3, 4, 5], 3, 5) == [1, 2, 3]
    assert fia_oracle.resolve_lengths(None, 2, 7) == [7, 7]
    with pytest.raises(ValueError):
        fia_oracle.resolve_lengths([1, 2], 3, 5)
    with pytest.raises(ValueError):
        fia_oracle.resolve_lengths([6], 1, 5)
    assert fia_oracle.tnd_lengths([3, 3, 10]) == ([0, 3, 3], [3, 0, 7])
    with pytest.raises(ValueError):
        fia_oracle.tnd_lengths([3, 2])

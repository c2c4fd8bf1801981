"""Comparison helpers for the GPU parity tests.

Tolerances are the ones the operator is held to: attention_out max-abs error
4e-3 for fp16 outputs and 1.6e-2 for bf16 outputs; softmax_lse within
1e-3 * max(1, |lse|); +inf LSE entries (rows without keys) must match exactly.
"""
import os

import numpy as np
import torch

OUT_TOL = {torch.float16: 4e-3, torch.bfloat16: 1.6e-2}
LSE_REL = 1e-3


def out_tol(dtype):
    return OUT_TOL[dtype]


def _record(what, value):
    """Appends a measured error to the file FIA_PARITY_LOG names (if set)."""
    path = os.environ.get("FIA_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(f"{os.environ.get('PYTEST_CURRENT_TEST', '?').split(' ')[0]}\t{what}\t{float(value):.3e}\n")


def assert_out_close(gpu, ref, dtype, what="attention_out"):
    g = gpu.detach().float().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    assert np.all(np.isfinite(g)), f"{what}: non-finite values"
    err = np.abs(g - ref).max() if g.size else 0.0
    _record(what + " max abs", err)
    assert err <= OUT_TOL[dtype], f"{what}: max abs err {err:.3e} > {OUT_TOL[dtype]:.1e}"
    return err


def assert_lse_close(gpu, ref, what="softmax_lse"):
    g = gpu.detach().cpu().numpy().astype(np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert g.shape == ref.shape, f"{what}: shape {g.shape} vs {ref.shape}"
    inf_ref = np.isinf(ref)
    assert np.array_equal(np.isinf(g) & (g > 0), inf_ref & (ref > 0)), f"{what}: +inf pattern differs"
    fin = ~inf_ref
    if fin.any():
        rel = np.abs(g[fin] - ref[fin]) / np.maximum(1.0, np.abs(ref[fin]))
        _record(what + " max rel", rel.max())
        assert rel.max() <= LSE_REL, f"{what}: rel err {rel.max():.3e} > {LSE_REL:.0e}"
        return rel.max()
    return 0.0


def assert_rows_close(gpu_out, gpu_lse, rows, ref_rows, index, dtype):
    """Sampled-row comparison: index(row) -> tuple indexing one output row."""
    tol = OUT_TOL[dtype]
    worst = 0.0
    worst_lse = 0.0
    for row, (o_ref, l_ref) in zip(rows, ref_rows):
        ix = index(row)
        g = gpu_out[ix].float().cpu().numpy().astype(np.float64)
        err = np.abs(g - o_ref).max()
        worst = max(worst, err)
        assert err <= tol, f"row {row}: max abs err {err:.3e} > {tol:.1e}"
        if gpu_lse is not None:
            gl = float(gpu_lse[ix][0]) if gpu_lse[ix].dim() else float(gpu_lse[ix])
            if np.isinf(l_ref):
                assert gl == float("inf"), f"row {row}: lse {gl} expected +inf"
            else:
                rel = abs(gl - l_ref) / max(1.0, abs(l_ref))
                worst_lse = max(worst_lse, rel)
                assert rel <= LSE_REL, f"row {row}: lse {gl} vs {l_ref}"
    _record("sampled rows max abs", worst)
    if gpu_lse is not None:
        _record("sampled rows lse max rel", worst_lse)
    return worst

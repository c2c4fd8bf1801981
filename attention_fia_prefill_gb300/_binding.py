"""ctypes binding of libfia (include/fia.h): argument marshalling only.

Every step of the attention runs in the library's CUDA kernels.  The functions
here turn torch tensors into fia_tensor descriptors, allocate outputs and the
workspace with torch on the tensors' device, and pass the current CUDA stream.
There is no fallback: a missing library or a failing call raises.
"""
from __future__ import annotations

import ctypes
import os

INT32_MAX = 2147483647
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libfia.so")

FIA_OK = 0
STATUS_NAMES = {
    0: "FIA_OK", 1: "FIA_ERR_NULL", 2: "FIA_ERR_DTYPE", 3: "FIA_ERR_SHAPE", 4: "FIA_ERR_LAYOUT",
    5: "FIA_ERR_UNSUPPORTED", 6: "FIA_ERR_SEQLEN", 7: "FIA_ERR_BLOCK_TABLE", 8: "FIA_ERR_WORKSPACE",
    9: "FIA_ERR_CUDA", 10: "FIA_ERR_TIMEOUT", 11: "FIA_ERR_HEADS", 12: "FIA_ERR_SPARSE_MODE",
    13: "FIA_ERR_ALIGNMENT",
}
DTYPE_F16, DTYPE_BF16, DTYPE_F32, DTYPE_I32, DTYPE_I64, DTYPE_U8, DTYPE_BOOL, DTYPE_I8, DTYPE_F8E4M3 = range(9)

# Every symbol include/fia.h declares.
EXPORTS = [
    "fia_params_init", "fia_prefill_get_workspace_size", "fia_prefill", "fia_prefill_mla_get_workspace_size",
    "fia_prefill_mla", "fia_prefill_paged_get_workspace_size", "fia_prefill_paged", "fia_decode_get_workspace_size",
    "fia_decode", "bsa_get_workspace_size", "bsa_forward", "bsa_fp8_get_workspace_size", "bsa_forward_fp8",
    "fia_device_status", "fia_status_string",
    "fia_last_error", "fia_profile_next_call", "fia_debug_set_wait_limit_ns", "fia_debug_set_decode_path", "fia_decode_no_alloc",
    "fia_debug_plan_decode",
]


class FIAError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {detail}")


class FiaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 5)]


class FiaParams(ctypes.Structure):
    _fields_ = [
        ("num_heads", ctypes.c_int64), ("num_key_value_heads", ctypes.c_int64), ("scale_value", ctypes.c_double),
        ("input_layout", ctypes.c_char_p), ("sparse_mode", ctypes.c_int64), ("pre_tokens", ctypes.c_int64),
        ("next_tokens", ctypes.c_int64), ("actual_seq_qlen", ctypes.POINTER(ctypes.c_int64)),
        ("n_actual_seq_qlen", ctypes.c_int64), ("actual_seq_kvlen", ctypes.POINTER(ctypes.c_int64)),
        ("n_actual_seq_kvlen", ctypes.c_int64), ("block_size", ctypes.c_int64),
        ("softmax_lse_flag", ctypes.c_int32), ("inner_precise", ctypes.c_int32),
    ]


_lib = None


def load_library(path: str | None = None):
    """Loads libfia.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise ImportError(f"libfia.so not built at {p}; run attention_fia_prefill_gb300.build.build()")
    lib = ctypes.CDLL(p)
    T = ctypes.POINTER(FiaTensor)
    P = ctypes.POINTER(FiaParams)
    st = ctypes.c_int
    sz = ctypes.POINTER(ctypes.c_size_t)
    vp = ctypes.c_void_p
    lib.fia_params_init.argtypes = [P]
    lib.fia_params_init.restype = None
    lib.fia_prefill_get_workspace_size.argtypes = [T, T, T, T, P, T, T, sz]
    lib.fia_prefill_get_workspace_size.restype = st
    lib.fia_prefill.argtypes = [T, T, T, T, P, T, T, vp, ctypes.c_size_t, vp]
    lib.fia_prefill.restype = st
    lib.fia_prefill_mla_get_workspace_size.argtypes = [T, T, T, T, T, T, P, T, T, sz]
    lib.fia_prefill_mla_get_workspace_size.restype = st
    lib.fia_prefill_mla.argtypes = [T, T, T, T, T, T, P, T, T, vp, ctypes.c_size_t, vp]
    lib.fia_prefill_mla.restype = st
    lib.fia_prefill_paged_get_workspace_size.argtypes = [T, T, T, T, T, P, T, T, sz]
    lib.fia_prefill_paged_get_workspace_size.restype = st
    lib.fia_prefill_paged.argtypes = [T, T, T, T, T, P, T, T, vp, ctypes.c_size_t, vp]
    lib.fia_prefill_paged.restype = st
    lib.fia_decode_get_workspace_size.argtypes = [T, T, T, T, T, T, T, P, T, T, sz]
    lib.fia_decode_get_workspace_size.restype = st
    lib.fia_decode.argtypes = [T, T, T, T, T, T, T, P, T, T, vp, ctypes.c_size_t, vp]
    lib.fia_decode.restype = st
    lib.bsa_get_workspace_size.argtypes = [T, T, T, T, ctypes.POINTER(ctypes.c_int64), P, T, T, sz]
    lib.bsa_get_workspace_size.restype = st
    lib.bsa_forward.argtypes = [T, T, T, T, ctypes.POINTER(ctypes.c_int64), P, T, T, vp, ctypes.c_size_t, vp]
    lib.bsa_forward.restype = st
    lib.bsa_fp8_get_workspace_size.argtypes = [T, T, T, T, ctypes.POINTER(ctypes.c_int64), T, T, T, P, T, T, sz]
    lib.bsa_fp8_get_workspace_size.restype = st
    lib.bsa_forward_fp8.argtypes = [T, T, T, T, ctypes.POINTER(ctypes.c_int64), T, T, T, P, T, T, vp,
                                    ctypes.c_size_t, vp]
    lib.bsa_forward_fp8.restype = st
    lib.fia_device_status.argtypes = [vp, vp]
    lib.fia_device_status.restype = st
    lib.fia_status_string.argtypes = [st]
    lib.fia_status_string.restype = ctypes.c_char_p
    lib.fia_last_error.argtypes = []
    lib.fia_last_error.restype = ctypes.c_char_p
    lib.fia_profile_next_call.argtypes = [vp, vp]
    lib.fia_profile_next_call.restype = None
    lib.fia_debug_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.fia_debug_set_wait_limit_ns.restype = None
    lib.fia_debug_set_decode_path.argtypes = [ctypes.c_int]
    lib.fia_debug_set_decode_path.restype = None
    lib.fia_decode_no_alloc.argtypes = [T, T, T, T, T, T, T, P, T, T, vp]
    lib.fia_decode_no_alloc.restype = st
    i32p, ip = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int)
    lib.fia_debug_plan_decode.argtypes = [i32p, ctypes.c_int, ctypes.c_int, ctypes.c_int, i32p, ctypes.c_int, i32p,
                                          ctypes.c_int, i32p, ctypes.c_int, ip, ip]
    lib.fia_debug_plan_decode.restype = st
    if path is None:
        _lib = lib
    return lib


# ------------------------------------------------------------------ marshalling
_DTYPE_CODES = None
_SHAPE5 = ctypes.c_int64 * 5


def _dtype_code(t) -> int:
    global _DTYPE_CODES
    if _DTYPE_CODES is None:
        import torch
        _DTYPE_CODES = {torch.float16: DTYPE_F16, torch.bfloat16: DTYPE_BF16, torch.float32: DTYPE_F32,
                        torch.int32: DTYPE_I32, torch.int64: DTYPE_I64, torch.uint8: DTYPE_U8, torch.bool: DTYPE_BOOL,
                        torch.int8: DTYPE_I8, torch.float8_e4m3fn: DTYPE_F8E4M3}
    code = _DTYPE_CODES.get(t.dtype)
    if code is None:
        raise TypeError(f"unsupported dtype {t.dtype}")
    return code


# Descriptors of recent tensors by (address, dtype, shape): a decode loop
# passes the same buffers call after call, and building the ctypes struct is
# most of a descriptor's cost.  The callee only reads a descriptor.
_DESC_CACHE: dict = {}


def tensor_desc(t) -> FiaTensor | None:
    """fia_tensor for a contiguous torch tensor (None stays None)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    shape = t.shape
    key = (t.data_ptr(), t.dtype, shape)
    d = _DESC_CACHE.get(key)
    if d is not None:
        return d
    if len(shape) > 5:
        raise ValueError("at most 5 dims")
    d = FiaTensor(key[0] or None, _dtype_code(t), len(shape), _SHAPE5(*shape))
    if len(_DESC_CACHE) >= 64:
        _DESC_CACHE.pop(next(iter(_DESC_CACHE)))
    _DESC_CACHE[key] = d
    return d


def raw_desc(ptr: int | None, dtype: int, shape) -> FiaTensor:
    """fia_tensor from a raw pointer (used by host-only validation tests)."""
    d = FiaTensor()
    d.data = ptr
    d.dtype = dtype
    d.ndim = len(shape)
    for i, s in enumerate(shape):
        d.shape[i] = int(s)
    return d


def _ref(d):
    return ctypes.byref(d) if d is not None else None


class Params:
    """Builds an fia_params struct; keeps the host length arrays alive."""

    def __init__(self, *, num_heads, num_key_value_heads=0, scale_value=1.0, input_layout="BSH", sparse_mode=0,
                 pre_tokens=INT32_MAX, next_tokens=INT32_MAX, actual_seq_qlen=None, actual_seq_kvlen=None,
                 block_size=0, softmax_lse_flag=False, inner_precise=0):
        self._layout = input_layout.encode()
        self._q = self._kv = None
        nq = nkv = 0
        if actual_seq_qlen is not None:
            nq = len(actual_seq_qlen)
            self._q = (ctypes.c_int64 * nq)(*actual_seq_qlen)
        if actual_seq_kvlen is not None:
            nkv = len(actual_seq_kvlen)
            self._kv = (ctypes.c_int64 * nkv)(*actual_seq_kvlen)
        I64P = ctypes.POINTER(ctypes.c_int64)
        self.p = FiaParams(int(num_heads), int(num_key_value_heads), float(scale_value), self._layout,
                           int(sparse_mode), int(pre_tokens), int(next_tokens),
                           ctypes.cast(self._q, I64P) if self._q is not None else None, nq,
                           ctypes.cast(self._kv, I64P) if self._kv is not None else None, nkv,
                           int(block_size), 1 if softmax_lse_flag else 0, int(inner_precise))


# The parameters of the last few calls, by value: a decode loop calls with the
# same lengths for every layer of a step, so the struct is built once per step.
_PARAMS_CACHE: dict = {}


def _params(**kw) -> Params:
    key = tuple((k, tuple(v) if isinstance(v, list) else v) for k, v in kw.items())
    try:
        prm = _PARAMS_CACHE.get(key)
    except TypeError:   # unhashable argument (e.g. a tensor of lengths): no caching
        return Params(**kw)
    if prm is None:
        if len(_PARAMS_CACHE) >= 16:
            _PARAMS_CACHE.pop(next(iter(_PARAMS_CACHE)))
        prm = _PARAMS_CACHE[key] = Params(**kw)
    return prm


def check(status: int):
    if status != FIA_OK:
        lib = load_library()
        raise FIAError(status, lib.fia_last_error().decode(errors="replace"))


_RAW_STREAM = None


def _stream_ptr(device):
    """The device's current CUDA stream (torch's raw accessor when it has one:
    a tenth of the cost of building a torch.cuda.Stream object)."""
    global _RAW_STREAM
    import torch
    if _RAW_STREAM is None:
        _RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", False)
    if _RAW_STREAM:
        idx = device.index if device.index is not None else torch.cuda.current_device()
        return ctypes.c_void_p(_RAW_STREAM(idx))
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


FIA_ERR_WORKSPACE = 8


def _run_with_workspace(size_fn, run_fn, args, workspace, device):
    """Runs run_fn(*args, ws, ws_bytes, stream).  A caller workspace is tried
    first (the call itself checks its size); otherwise, or when it is too
    small, the size is queried and a workspace allocated with torch."""
    stream = _stream_ptr(device)
    if workspace is not None:
        st = run_fn(*args, ctypes.c_void_p(workspace.data_ptr()), ctypes.c_size_t(workspace.numel()), stream)
        if st != FIA_ERR_WORKSPACE:
            check(st)
            return
    import torch
    ws = ctypes.c_size_t(0)
    check(size_fn(*args, ctypes.byref(ws)))
    workspace = torch.empty(max(ws.value, 1), dtype=torch.uint8, device=device)
    check(run_fn(*args, ctypes.c_void_p(workspace.data_ptr()), ctypes.c_size_t(workspace.numel()), stream))


def _lse_shape(q, layout, num_heads):
    if layout == "TND":
        return (q.shape[0], num_heads, 1)
    if layout == "BNSD":
        return (q.shape[0], num_heads, q.shape[2], 1)
    return (q.shape[0], num_heads, q.shape[1], 1)


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("fia kernels take CUDA tensors")


# ------------------------------------------------------------------ public API
def fia_prefill(query, key, value, *, atten_mask=None, actual_seq_qlen=None, actual_seq_kvlen=None, num_heads=1,
                num_key_value_heads=0, scale_value=1.0, input_layout="BSH", sparse_mode=0, pre_tokens=INT32_MAX,
                next_tokens=INT32_MAX, softmax_lse_flag=False, inner_precise=0, out=None, softmax_lse=None,
                workspace=None):
    """Full attention (Q_S >= 1).  Returns (attention_out, softmax_lse or None)."""
    import torch
    _require_cuda(query, key, value, atten_mask)
    lib = load_library()
    prm = _params(num_heads=num_heads, num_key_value_heads=num_key_value_heads, scale_value=scale_value,
                 input_layout=input_layout, sparse_mode=sparse_mode, pre_tokens=pre_tokens, next_tokens=next_tokens,
                 actual_seq_qlen=actual_seq_qlen, actual_seq_kvlen=actual_seq_kvlen,
                 softmax_lse_flag=softmax_lse_flag, inner_precise=inner_precise)
    if out is None:
        out = torch.empty_like(query)
    if softmax_lse_flag and softmax_lse is None:
        softmax_lse = torch.empty(_lse_shape(query, input_layout, num_heads), dtype=torch.float32, device=query.device)
    dq, dk, dv, dm, do, dl = (tensor_desc(t) for t in (query, key, value, atten_mask, out, softmax_lse))
    _run_with_workspace(lib.fia_prefill_get_workspace_size, lib.fia_prefill,
                        (_ref(dq), _ref(dk), _ref(dv), _ref(dm), ctypes.byref(prm.p), _ref(do), _ref(dl)),
                        workspace, query.device)
    return out, softmax_lse


def fia_prefill_mla(query, key, value, *, query_rope=None, key_rope=None, atten_mask=None, actual_seq_qlen=None,
                    actual_seq_kvlen=None, num_heads=1, num_key_value_heads=0, scale_value=1.0, input_layout="TND",
                    sparse_mode=0, pre_tokens=INT32_MAX, next_tokens=INT32_MAX, softmax_lse_flag=False,
                    inner_precise=0, out=None, softmax_lse=None, workspace=None):
    """MLA prefill: query/key D 192 (or D 128 with query_rope / key_rope of D 64),
    value D 128.  Returns (attention_out with value's head dim, softmax_lse or None)."""
    import torch
    _require_cuda(query, key, value, query_rope, key_rope, atten_mask)
    lib = load_library()
    prm = _params(num_heads=num_heads, num_key_value_heads=num_key_value_heads, scale_value=scale_value,
                 input_layout=input_layout, sparse_mode=sparse_mode, pre_tokens=pre_tokens, next_tokens=next_tokens,
                 actual_seq_qlen=actual_seq_qlen, actual_seq_kvlen=actual_seq_kvlen,
                 softmax_lse_flag=softmax_lse_flag, inner_precise=inner_precise)
    if out is None:
        nkv = num_key_value_heads or num_heads
        dv = value.shape[-1] // nkv if input_layout == "BSH" else value.shape[-1]
        shape = list(query.shape)
        shape[-1] = num_heads * dv if input_layout == "BSH" else dv
        out = torch.empty(shape, dtype=query.dtype, device=query.device)
    if softmax_lse_flag and softmax_lse is None:
        softmax_lse = torch.empty(_lse_shape(query, input_layout, num_heads), dtype=torch.float32, device=query.device)
    descs = [tensor_desc(t) for t in (query, key, value, query_rope, key_rope, atten_mask, out, softmax_lse)]
    dq, dk, dv_, dqr, dkr, dm, do, dl = (_ref(d) for d in descs)
    _run_with_workspace(lib.fia_prefill_mla_get_workspace_size, lib.fia_prefill_mla,
                        (dq, dk, dv_, dqr, dkr, dm, ctypes.byref(prm.p), do, dl), workspace, query.device)
    return out, softmax_lse


def fia_prefill_paged(query, key_cache, value_cache, block_table, *, block_size, actual_seq_kvlen, atten_mask=None,
                      actual_seq_qlen=None, num_heads=1, num_key_value_heads=0, scale_value=1.0, input_layout="BSH",
                      sparse_mode=0, pre_tokens=INT32_MAX, next_tokens=INT32_MAX, softmax_lse_flag=False,
                      inner_precise=0, out=None, softmax_lse=None, workspace=None):
    """Prefill (any Q_S) against a paged KV cache: key_cache / value_cache are
    (blocknum, KV_N, block_size, D) or (blocknum, block_size, KV_N*D) pools,
    block_table int32 (B, max blocks), actual_seq_kvlen per-batch key counts.
    Returns (attention_out, softmax_lse or None)."""
    import torch
    _require_cuda(query, key_cache, value_cache, block_table, atten_mask)
    lib = load_library()
    prm = _params(num_heads=num_heads, num_key_value_heads=num_key_value_heads, scale_value=scale_value,
                 input_layout=input_layout, sparse_mode=sparse_mode, pre_tokens=pre_tokens, next_tokens=next_tokens,
                 actual_seq_qlen=actual_seq_qlen, actual_seq_kvlen=actual_seq_kvlen, block_size=block_size,
                 softmax_lse_flag=softmax_lse_flag, inner_precise=inner_precise)
    if out is None:
        out = torch.empty_like(query)
    if softmax_lse_flag and softmax_lse is None:
        softmax_lse = torch.empty(_lse_shape(query, input_layout, num_heads), dtype=torch.float32, device=query.device)
    descs = [tensor_desc(t) for t in (query, key_cache, value_cache, block_table, atten_mask, out, softmax_lse)]
    dq, dk, dv, dt, dm, do, dl = (_ref(d) for d in descs)
    _run_with_workspace(lib.fia_prefill_paged_get_workspace_size, lib.fia_prefill_paged,
                        (dq, dk, dv, dt, dm, ctypes.byref(prm.p), do, dl), workspace, query.device)
    return out, softmax_lse


def fia_decode(query, key, value, *, query_rope=None, key_rope=None, block_table=None, block_size=0,
               actual_seq_kvlen=None, atten_mask=None, num_heads=1, num_key_value_heads=0, scale_value=1.0,
               input_layout="BSH", sparse_mode=0, softmax_lse_flag=False, inner_precise=0, out=None,
               softmax_lse=None, workspace=None):
    """Incremental attention against a paged or contiguous cache, optionally
    MLA.  Q_S = 1, or up to 16 new tokens per sequence (sparse_mode 0, 2 or 3
    over the Q_S x S_kv block; 3 = each token sees the cache up to itself)."""
    import torch
    _require_cuda(query, key, value, query_rope, key_rope, block_table)
    lib = load_library()
    prm = _params(num_heads=num_heads, num_key_value_heads=num_key_value_heads, scale_value=scale_value,
                 input_layout=input_layout, sparse_mode=sparse_mode, actual_seq_kvlen=actual_seq_kvlen,
                 block_size=block_size, softmax_lse_flag=softmax_lse_flag, inner_precise=inner_precise)
    if out is None:
        out = torch.empty_like(query)
    if softmax_lse_flag and softmax_lse is None:
        softmax_lse = torch.empty(_lse_shape(query, input_layout, num_heads), dtype=torch.float32, device=query.device)
    descs = [tensor_desc(t) for t in (query, key, value, query_rope, key_rope, block_table, atten_mask, out,
                                      softmax_lse)]
    dq, dk, dv, dqr, dkr, dbt, dm, do, dl = descs
    _run_with_workspace(lib.fia_decode_get_workspace_size, lib.fia_decode,
                        (_ref(dq), _ref(dk), _ref(dv), _ref(dqr), _ref(dkr), _ref(dbt), _ref(dm), ctypes.byref(prm.p),
                         _ref(do), _ref(dl)), workspace, query.device)
    return out, softmax_lse


def fia_decode_no_alloc(query, key, value, *, out, softmax_lse=None, query_rope=None, key_rope=None,
                        block_table=None, block_size=0, actual_seq_kvlen=None, atten_mask=None, num_heads=1,
                        num_key_value_heads=0, scale_value=1.0, input_layout="BSH", sparse_mode=0,
                        inner_precise=0):
    """fia_decode for callers that cannot allocate device memory: the caller
    passes every output buffer and the library supplies the scratch from its
    built-in array (see include/fia.h).  Nothing is allocated here."""
    _require_cuda(query, key, value, query_rope, key_rope, block_table, out, softmax_lse)
    lib = load_library()
    prm = _params(num_heads=num_heads, num_key_value_heads=num_key_value_heads, scale_value=scale_value,
                 input_layout=input_layout, sparse_mode=sparse_mode, actual_seq_kvlen=actual_seq_kvlen,
                 block_size=block_size, softmax_lse_flag=softmax_lse is not None, inner_precise=inner_precise)
    descs = [tensor_desc(t) for t in (query, key, value, query_rope, key_rope, block_table, atten_mask, out,
                                      softmax_lse)]
    dq, dk, dv, dqr, dkr, dbt, dm, do, dl = descs
    check(lib.fia_decode_no_alloc(_ref(dq), _ref(dk), _ref(dv), _ref(dqr), _ref(dkr), _ref(dbt), _ref(dm),
                                  ctypes.byref(prm.p), _ref(do), _ref(dl), _stream_ptr(query.device)))
    return out, softmax_lse


def bsa_forward(query, key, value, block_sparse_mask, block_shape, *, actual_seq_qlen=None, actual_seq_kvlen=None,
                num_heads=1, num_key_value_heads=0, scale_value=1.0, input_layout="BNSD", softmax_lse_flag=False,
                out=None, softmax_lse=None, workspace=None, q_dequant_scale=None, k_dequant_scale=None,
                v_dequant_scale=None):
    """Block-sparse attention: each query block attends to the KV blocks its mask row keeps.
    With float8 e4m3 query/key/value pass the three fp32 dequant scales (FP8
    path, bf16 output)."""
    import torch
    fp8 = q_dequant_scale is not None or k_dequant_scale is not None or v_dequant_scale is not None
    _require_cuda(query, key, value, block_sparse_mask, q_dequant_scale, k_dequant_scale, v_dequant_scale)
    lib = load_library()
    prm = _params(num_heads=num_heads, num_key_value_heads=num_key_value_heads, scale_value=scale_value,
                 input_layout=input_layout, actual_seq_qlen=actual_seq_qlen, actual_seq_kvlen=actual_seq_kvlen,
                 softmax_lse_flag=softmax_lse_flag)
    if out is None:
        out = torch.empty(query.shape, dtype=torch.bfloat16 if fp8 else query.dtype, device=query.device)
    if softmax_lse_flag and softmax_lse is None:
        softmax_lse = torch.empty(_lse_shape(query, input_layout, num_heads), dtype=torch.float32, device=query.device)
    shape = (ctypes.c_int64 * 2)(int(block_shape[0]), int(block_shape[1]))
    dq, dk, dv, dmask, do, dl = (tensor_desc(t) for t in (query, key, value, block_sparse_mask, out, softmax_lse))
    if fp8:
        dsq, dsk, dsv = (_ref(tensor_desc(t)) for t in (q_dequant_scale, k_dequant_scale, v_dequant_scale))
        _run_with_workspace(lib.bsa_fp8_get_workspace_size, lib.bsa_forward_fp8,
                            (_ref(dq), _ref(dk), _ref(dv), _ref(dmask), shape, dsq, dsk, dsv, ctypes.byref(prm.p),
                             _ref(do), _ref(dl)), workspace, query.device)
    else:
        _run_with_workspace(lib.bsa_get_workspace_size, lib.bsa_forward,
                            (_ref(dq), _ref(dk), _ref(dv), _ref(dmask), shape, ctypes.byref(prm.p), _ref(do),
                             _ref(dl)), workspace, query.device)
    return out, softmax_lse


def debug_plan_decode(kv_len, num_key_value_heads, n_cta_max):
    """The decode plan the library deals (host only): returns (cta_seg of
    n_cta + 1 entries, segs as rows (unit, stage_begin, stage_end, part),
    unit_parts as rows (first part, parts)) as lists."""
    lib = load_library()
    B, N2 = len(kv_len), int(num_key_value_heads)
    n_units = B * N2
    cap_cta, cap_segs = int(n_cta_max) + 1, 4 * (n_units + int(n_cta_max) + 1)
    lens = (ctypes.c_int32 * max(B, 1))(*[int(x) for x in kv_len])
    cta_seg = (ctypes.c_int32 * cap_cta)()
    segs = (ctypes.c_int32 * cap_segs)()
    parts = (ctypes.c_int32 * max(2 * n_units, 1))()
    n_cta, n_segs = ctypes.c_int(0), ctypes.c_int(0)
    check(lib.fia_debug_plan_decode(lens, B, N2, int(n_cta_max), cta_seg, cap_cta, segs, cap_segs, parts,
                                    max(2 * n_units, 1), ctypes.byref(n_cta), ctypes.byref(n_segs)))
    return (list(cta_seg[:n_cta.value + 1]), [tuple(segs[4 * i:4 * i + 4]) for i in range(n_segs.value)],
            [tuple(parts[2 * u:2 * u + 2]) for u in range(n_units)])


def profile_next_call(start_event, stop_event):
    """Record two torch.cuda.Event objects around the main kernel of the next call."""
    lib = load_library()
    lib.fia_profile_next_call(ctypes.c_void_p(start_event.cuda_event), ctypes.c_void_p(stop_event.cuda_event))


def fia_device_status(workspace) -> int:
    """Device-side status recorded in a workspace (synchronises the current stream)."""
    lib = load_library()
    return lib.fia_device_status(ctypes.c_void_p(workspace.data_ptr()), _stream_ptr(workspace.device))

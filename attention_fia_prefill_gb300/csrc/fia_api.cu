// Host side of the C ABI declared in include/fia.h: argument validation,
// per-batch length resolution, work planning, TMA descriptor encoding, and the
// kernel launches.  Nothing here allocates device memory: plans and partial
// results live in the caller's workspace.
#include "../../include/fia.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

using namespace fia;

namespace {

thread_local std::string g_last_error;

// Events the caller asked to have recorded around the main kernel of its next
// call on this thread (fia_profile_next_call).
thread_local cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

template <typename F>
cudaError_t profiled(cudaStream_t s, F&& launch) {
  cudaEvent_t a = g_prof_start, b = g_prof_stop;
  g_prof_start = g_prof_stop = nullptr;
  if (a != nullptr) {
    cudaError_t e = cudaEventRecord(a, s);
    if (e != cudaSuccess) return e;
  }
  cudaError_t e = launch();
  if (e != cudaSuccess) return e;
  if (b != nullptr) return cudaEventRecord(b, s);
  return cudaSuccess;
}

fia_status fail(fia_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return s;
}

constexpr int64_t kInt32Max = 2147483647;
constexpr size_t kHeader = 256;   // workspace bytes [0, 256): device status word + padding

// Every call gets a fresh epoch; kernels tag the workspace's status word (and
// the decode kernel its per-unit counters) with it, so nothing in a reused
// workspace has to be cleared between calls.
std::atomic<unsigned long long> g_epoch{0};
unsigned long long next_epoch() { return g_epoch.fetch_add(1, std::memory_order_relaxed) + 1; }

// Limit of the kernels' unwinding waits (fia_debug_set_wait_limit_ns; 0: the
// default of kWaitLimitNs).
std::atomic<unsigned long long> g_wait_limit_ns{0};
// fia_debug_set_decode_path: 1 runs the tcgen05 decode kernel for every unit
std::atomic<int> g_decode_force_tc{0};

// A call's device status: the word at the start of its workspace, a fresh
// epoch, and the wait limit.
DevStatus make_status(void* workspace) {
  const unsigned long long lim = g_wait_limit_ns.load(std::memory_order_relaxed);
  return DevStatus{reinterpret_cast<unsigned long long*>(workspace), next_epoch(), lim != 0 ? lim : kWaitLimitNs};
}

// Status word for calls that launch no stamping kernel: cleared on the stream.
fia_status clear_status(void* ws, cudaStream_t stream);
constexpr int kMaxDecodeCtas = 256;   // decode CTAs per call (one per SM)

int64_t numel(const fia_tensor* t) {
  if (t == nullptr || t->ndim <= 0) return 0;
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}

// An optional tensor is present when it has a rank and data.  A required tensor
// may have no data when it holds zero elements (e.g. K/V with S2 = 0).
bool present(const fia_tensor* t) { return t != nullptr && t->data != nullptr && t->ndim > 0; }
bool given(const fia_tensor* t) {
  return t != nullptr && t->ndim > 0 && (t->data != nullptr || numel(t) == 0);
}

bool is_half(int32_t dt) { return dt == FIA_DTYPE_F16 || dt == FIA_DTYPE_BF16; }

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

enum Layout { L_BSH, L_BSND, L_BNSD, L_TND, L_BAD };

Layout parse_layout(const char* s) {
  if (s == nullptr) return L_BSH;
  if (!strcmp(s, "BSH")) return L_BSH;
  if (!strcmp(s, "BSND")) return L_BSND;
  if (!strcmp(s, "BNSD")) return L_BNSD;
  if (!strcmp(s, "TND")) return L_TND;
  return L_BAD;
}

// --------------------------------------------------------------- TMA encode
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// rank-d tiled map of 16-bit elements, 128-byte swizzle, box {64, box_rows, 1, ...}
// Boxes of 128 bytes x box_rows: 64 16-bit elements, or 128 8-bit ones (u8).
fia_status make_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims, const uint64_t* strides_bytes,
                    uint32_t box_rows, bool u8 = false) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return fail(FIA_ERR_CUDA, "cuTensorMapEncodeTiled unavailable (no CUDA driver?)");
  cuuint64_t gd[5], gs[4];
  cuuint32_t box[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    box[i] = i == 0 ? (u8 ? 128 : 64) : (i == 1 ? box_rows : 1);
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) gs[i] = strides_bytes[i];
  CUresult r = fn(m, u8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_UINT16, rank,
                  const_cast<void*>(base), gd, gs, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FIA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return FIA_OK;
}

fia_status cuda_check(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(FIA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
  return FIA_OK;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

// ------------------------------------------------------ length resolution
// actual_seq_* rules (npu_fused_infer_attention_score_v2, actual_seq_qlen /
// actual_seq_kvlen): absent -> the tensor's S; one entry -> every batch; >= B
// entries -> the first B; other counts are errors; entries in [0, S].
fia_status resolve_lengths(const int64_t* lst, int64_t n, int64_t B, int64_t S, std::vector<int32_t>& out,
                           const char* name) {
  out.assign(size_t(B), int32_t(S));
  if (lst == nullptr) {
    if (n != 0) return fail(FIA_ERR_SEQLEN, "%s: NULL list with nonzero count", name);
    return FIA_OK;
  }
  if (n != 1 && n < B) return fail(FIA_ERR_SEQLEN, "%s: %lld entries for B=%lld", name, (long long)n, (long long)B);
  for (int64_t b = 0; b < B; ++b) {
    const int64_t v = lst[n == 1 ? 0 : b];
    if (v < 0 || v > S) return fail(FIA_ERR_SEQLEN, "%s[%lld]=%lld outside [0,%lld]", name, (long long)b, (long long)v, (long long)S);
    out[size_t(b)] = int32_t(v);
  }
  return FIA_OK;
}

// TND: cumulative lengths without a leading 0; B = list length (<= 4096),
// non-decreasing, non-negative, last entry <= T.
fia_status resolve_tnd(const int64_t* lst, int64_t n, int64_t T, std::vector<int32_t>& start,
                       std::vector<int32_t>& len, const char* name) {
  if (lst == nullptr || n <= 0) return fail(FIA_ERR_SEQLEN, "%s is required for TND", name);
  if (n > 4096) return fail(FIA_ERR_SEQLEN, "%s has %lld entries (> 4096)", name, (long long)n);
  start.resize(size_t(n));
  len.resize(size_t(n));
  int64_t prev = 0;
  for (int64_t b = 0; b < n; ++b) {
    if (lst[b] < prev) return fail(FIA_ERR_SEQLEN, "%s must be non-decreasing and non-negative", name);
    start[size_t(b)] = int32_t(prev);
    len[size_t(b)] = int32_t(lst[b] - prev);
    prev = lst[b];
  }
  if (prev > T) return fail(FIA_ERR_SEQLEN, "%s total %lld exceeds T=%lld", name, (long long)prev, (long long)T);
  return FIA_OK;
}

// GQA rules (num_key_value_heads): Q_N a multiple of KV_N, Q_N / KV_N <= 64.
// The MLA case (query_rope/key_rope given) takes Q_N up to 128 over KV_N = 1.
fia_status resolve_heads(const fia_params* p, int64_t& N1, int64_t& N2, int64_t max_ratio = 64) {
  N1 = p->num_heads;
  N2 = p->num_key_value_heads == 0 ? p->num_heads : p->num_key_value_heads;
  if (N1 <= 0 || N2 <= 0) return fail(FIA_ERR_HEADS, "num_heads=%lld num_key_value_heads=%lld", (long long)N1, (long long)N2);
  if (N1 % N2 != 0) return fail(FIA_ERR_HEADS, "num_heads %lld not a multiple of num_key_value_heads %lld", (long long)N1, (long long)N2);
  if (N1 / N2 > max_ratio)
    return fail(FIA_ERR_HEADS, "num_heads / num_key_value_heads = %lld > %lld", (long long)(N1 / N2), (long long)max_ratio);
  return FIA_OK;
}

// ------------------------------------------------------------ prefill plan
struct Geometry {
  Layout layout;
  int64_t B, N1, N2, S1, S2, D, T1, T2;
  bool bf16;
  std::vector<BatchInfo> batches;
  int band_pre = 0, band_next = 0;   // sparse_mode 4 / explicit mask, clamped to +-2^30
  // explicit atten_mask (sparse_mode 0 with a mask, 1)
  const uint8_t* mask = nullptr;
  int64_t mask_sb = 0, mask_ss = 0;
  int64_t mask_s1 = 0;               // rows of one mask slice (its key extent is mask_ss)
  int mask_cs = 1;
  // head dims the kernels run with: scores over Dqk, value / output Dv (MLA
  // prefill: 192 / 128, with the rope columns from qr / kr when given)
  int64_t Dqk = 0, Dv = 0;
  bool mla = false;
  bool fp8 = false;   // FP8 block-sparse: e4m3 query / key / value, bf16 output
  const float* fp8_q = nullptr;
  const float* fp8_k = nullptr;
  const float* fp8_v = nullptr;
  int fp8_nqs = 0, fp8_nks = 0;
  const fia_tensor* qr = nullptr;
  const fia_tensor* kr = nullptr;
  // paged K/V (chunked prefill): pools (blocknum, KV_N, bs, D) or (blocknum, bs, KV_N*D)
  bool paged = false, kv_bnbd = false;
  int64_t bs = 0, nblk = 0, table_stride = 0;
  const int32_t* table = nullptr;
};

// Shapes of q/k/v in a dense layout -> (B, N, S, D).  BSH splits H by heads.
fia_status dense_dims(const fia_tensor* t, Layout L, int64_t N, int64_t& B, int64_t& S, int64_t& D, const char* name) {
  if (L == L_BNSD || L == L_BSND) {
    if (t->ndim != 4) return fail(FIA_ERR_SHAPE, "%s must be 4-D for %s", name, L == L_BNSD ? "BNSD" : "BSND");
    B = t->shape[0];
    const int64_t n = L == L_BNSD ? t->shape[1] : t->shape[2];
    S = L == L_BNSD ? t->shape[2] : t->shape[1];
    D = t->shape[3];
    if (n != N) return fail(FIA_ERR_HEADS, "%s has %lld heads, expected %lld", name, (long long)n, (long long)N);
  } else if (L == L_BSH) {
    if (t->ndim != 3) return fail(FIA_ERR_SHAPE, "%s must be 3-D for BSH", name);
    B = t->shape[0];
    S = t->shape[1];
    if (t->shape[2] % N != 0) return fail(FIA_ERR_SHAPE, "%s H=%lld not divisible by %lld heads", name, (long long)t->shape[2], (long long)N);
    D = t->shape[2] / N;
  } else {
    if (t->ndim != 3) return fail(FIA_ERR_SHAPE, "%s must be 3-D for TND", name);
    B = -1;
    S = t->shape[0];
    if (t->shape[1] != N) return fail(FIA_ERR_HEADS, "%s has %lld heads, expected %lld", name, (long long)t->shape[1], (long long)N);
    D = t->shape[2];
  }
  return FIA_OK;
}

bool same_shape(const fia_tensor* a, const fia_tensor* b) {
  if (a->ndim != b->ndim) return false;
  for (int i = 0; i < a->ndim; ++i)
    if (a->shape[i] != b->shape[i]) return false;
  return true;
}

// Strides (elements) of (b, n, s) for a dense layout with N heads of D.
void bns_strides(Layout L, int64_t N, int64_t S, int64_t D, int64_t* st) {
  if (L == L_BNSD) { st[0] = N * S * D; st[1] = S * D; st[2] = D; }
  else if (L == L_TND) { st[0] = 0; st[1] = D; st[2] = N * D; }
  else { st[0] = S * N * D; st[1] = D; st[2] = N * D; }
}

fia_status check_lse(const fia_tensor* lse, const fia_params* p, Layout L, int64_t B, int64_t N1, int64_t S1, int64_t T1) {
  if (p->softmax_lse_flag == 0) return FIA_OK;
  if (!present(lse)) return fail(FIA_ERR_NULL, "softmax_lse_flag set but softmax_lse absent");
  if (lse->dtype != FIA_DTYPE_F32) return fail(FIA_ERR_DTYPE, "softmax_lse must be fp32");
  if (L == L_TND) {
    if (!(lse->ndim == 3 && lse->shape[0] == T1 && lse->shape[1] == N1 && lse->shape[2] == 1))
      return fail(FIA_ERR_SHAPE, "softmax_lse must be (T, N1, 1)");
  } else if (!(lse->ndim == 4 && lse->shape[0] == B && lse->shape[1] == N1 && lse->shape[2] == S1 && lse->shape[3] == 1)) {
    return fail(FIA_ERR_SHAPE, "softmax_lse must be (B, N1, S1, 1)");
  }
  if (!aligned16(lse->data)) return fail(FIA_ERR_ALIGNMENT, "softmax_lse not 16-byte aligned");
  return FIA_OK;
}

// Paged key/value pools for prefill (npu_fused_infer_attention_score_v2, page
// attention): block_table int32 (B, >= maxBlockNumPerSeq), block_size a
// multiple of 128 in 128..512, key/value (blocknum, KV_N, bs, D) or
// (blocknum, bs, KV_N*D) with the same shape.  Sets the pool fields and
// S2 = table columns x block_size; D of the key comes back in Dk.
fia_status paged_pools(const fia_tensor* k, const fia_tensor* v, const fia_tensor* table, const fia_params* p,
                       Geometry& g, int64_t& Dk) {
  if (table->dtype != FIA_DTYPE_I32 || table->ndim != 2)
    return fail(FIA_ERR_BLOCK_TABLE, "block_table must be int32 (B, maxBlocksPerSeq)");
  if (!aligned16(table->data)) return fail(FIA_ERR_ALIGNMENT, "block_table not 16-byte aligned");
  if (p->actual_seq_kvlen == nullptr) return fail(FIA_ERR_SEQLEN, "page attention needs actual_seq_kvlen");
  g.bs = p->block_size;
  if (g.bs < 128 || g.bs > 512 || g.bs % 128 != 0)
    return fail(FIA_ERR_BLOCK_TABLE, "block_size %lld: 128..512, a multiple of 128", (long long)g.bs);
  if (k->ndim == 4) {
    g.kv_bnbd = true;
    if (k->shape[1] != g.N2 || k->shape[2] != g.bs)
      return fail(FIA_ERR_SHAPE, "paged key must be (blocknum, KV_N, block_size, D)");
    Dk = k->shape[3];
  } else if (k->ndim == 3) {
    g.kv_bnbd = false;
    if (k->shape[1] != g.bs || k->shape[2] % g.N2 != 0)
      return fail(FIA_ERR_SHAPE, "paged key must be (blocknum, block_size, KV_N*D)");
    Dk = k->shape[2] / g.N2;
  } else {
    return fail(FIA_ERR_SHAPE, "paged key must be 3-D or 4-D");
  }
  g.paged = true;
  g.nblk = k->shape[0];
  g.table = static_cast<const int32_t*>(table->data);
  g.table_stride = table->shape[1];
  g.S2 = table->shape[1] * g.bs;
  return FIA_OK;
}

// Common validation of q/k/v/out for the dense prefill and block-sparse calls
// (and the paged prefill, with a block_table).
// MLA prefill (mla): value and output have D 128; query/key D 192, or D 128
// plus query_rope / key_rope of D 64.
fia_status prefill_geometry(const fia_tensor* q, const fia_tensor* k, const fia_tensor* v, const fia_params* p,
                            const fia_tensor* out, bool bsa, Geometry& g, const fia_tensor* table = nullptr,
                            bool mla = false, const fia_tensor* qr = nullptr, const fia_tensor* kr = nullptr,
                            bool fp8 = false) {
  if (p != nullptr) {
    const int64_t lim = int64_t(1) << 30;
    g.band_pre = int(std::max(-lim, std::min(lim, p->pre_tokens)));
    g.band_next = int(std::max(-lim, std::min(lim, p->next_tokens)));
  }
  if (p == nullptr) return fail(FIA_ERR_NULL, "params is NULL");
  if (!given(q) || !given(k) || !given(v) || !given(out))
    return fail(FIA_ERR_NULL, "query/key/value/attention_out required");
  g.layout = parse_layout(p->input_layout);
  if (g.layout == L_BAD) return fail(FIA_ERR_LAYOUT, "input_layout '%s' not supported", p->input_layout);
  if (bsa && g.layout == L_BSH) return fail(FIA_ERR_LAYOUT, "block-sparse attention takes TND, BNSD or BSND");
  if (fp8) {
    if (q->dtype != FIA_DTYPE_F8E4M3 || k->dtype != q->dtype || v->dtype != q->dtype)
      return fail(FIA_ERR_DTYPE, "FP8 attention takes float8 e4m3 query, key and value");
    if (out->dtype != FIA_DTYPE_BF16) return fail(FIA_ERR_DTYPE, "FP8 attention writes a bf16 attention_out");
  } else {
    if (!is_half(q->dtype) || k->dtype != q->dtype || v->dtype != q->dtype)
      return fail(FIA_ERR_DTYPE, "query/key/value must share fp16 or bf16");
    if (out->dtype != q->dtype) return fail(FIA_ERR_DTYPE, "attention_out must have the query's dtype");
  }
  g.fp8 = fp8;
  fia_status st = resolve_heads(p, g.N1, g.N2);
  if (st != FIA_OK) return st;
  if (!mla && !same_shape(k, v)) return fail(FIA_ERR_SHAPE, "key and value shapes differ");
  if (!mla && !same_shape(q, out)) return fail(FIA_ERR_SHAPE, "attention_out must have the query's shape");
  int64_t Bq, Bk, Dk;
  st = dense_dims(q, g.layout, g.N1, Bq, g.S1, g.D, "query");
  if (st != FIA_OK) return st;
  if (present(table)) {
    st = paged_pools(k, v, table, p, g, Dk);
    Bk = table->shape[0];
  } else {
    st = dense_dims(k, g.layout, g.N2, Bk, g.S2, Dk, "key");
  }
  if (st != FIA_OK) return st;
  if (Dk != g.D) return fail(FIA_ERR_SHAPE, "query D=%lld, key D=%lld", (long long)g.D, (long long)Dk);
  g.Dqk = g.Dv = g.D;
  if (mla) {
    if (present(table)) return fail(FIA_ERR_UNSUPPORTED, "MLA prefill takes contiguous key/value");
    int64_t Bv, Sv, Dv, Bo, So, Do;
    st = dense_dims(v, g.layout, g.N2, Bv, Sv, Dv, "value");
    if (st != FIA_OK) return st;
    st = dense_dims(out, g.layout, g.N1, Bo, So, Do, "attention_out");
    if (st != FIA_OK) return st;
    if (Bv != Bk || Sv != g.S2) return fail(FIA_ERR_SHAPE, "value must match key but for its head dim");
    if (Dv != 128) return fail(FIA_ERR_UNSUPPORTED, "MLA prefill takes value D 128 (got %lld)", (long long)Dv);
    if (Bo != Bq || So != g.S1 || Do != Dv)
      return fail(FIA_ERR_SHAPE, "attention_out must be the query's shape with value's head dim");
    if (present(qr) != present(kr)) return fail(FIA_ERR_SHAPE, "query_rope and key_rope must be given together");
    if (present(qr)) {
      if (g.D != 128) return fail(FIA_ERR_UNSUPPORTED, "with query_rope / key_rope, query and key take D 128");
      if (qr->dtype != q->dtype || kr->dtype != q->dtype) return fail(FIA_ERR_DTYPE, "rope tensors must match query");
      int64_t Br, Sr, Dr;
      st = dense_dims(qr, g.layout, g.N1, Br, Sr, Dr, "query_rope");
      if (st != FIA_OK) return st;
      if (Br != Bq || Sr != g.S1 || Dr != 64) return fail(FIA_ERR_SHAPE, "query_rope must be the query's shape with D 64");
      st = dense_dims(kr, g.layout, g.N2, Br, Sr, Dr, "key_rope");
      if (st != FIA_OK) return st;
      if (Br != Bk || Sr != g.S2 || Dr != 64) return fail(FIA_ERR_SHAPE, "key_rope must be the key's shape with D 64");
      if (!aligned16(qr->data) || !aligned16(kr->data)) return fail(FIA_ERR_ALIGNMENT, "rope tensors not 16-byte aligned");
    } else if (g.D != 192) {
      return fail(FIA_ERR_UNSUPPORTED, "MLA prefill takes query/key D 192, or D 128 with rope tensors (got %lld)",
                  (long long)g.D);
    }
    g.mla = true;
    g.qr = qr;
    g.kr = kr;
    g.Dqk = 192;
    g.Dv = 128;
  } else if (g.D != 64 && g.D != 128) {
    return fail(FIA_ERR_UNSUPPORTED, "head dim %lld (kernels take 64 or 128)", (long long)g.D);
  }
  if (fp8 && g.D != 128) return fail(FIA_ERR_UNSUPPORTED, "FP8 attention takes D 128 (got %lld)", (long long)g.D);
  if (!(p->scale_value > 0.0) || !std::isfinite(p->scale_value))
    return fail(FIA_ERR_UNSUPPORTED, "scale_value must be finite and > 0");
  if (p->inner_precise < 0 || p->inner_precise > 4) return fail(FIA_ERR_UNSUPPORTED, "inner_precise %d", p->inner_precise);
  g.bf16 = q->dtype == FIA_DTYPE_BF16 || fp8;
  if (!aligned16(q->data) || !aligned16(k->data) || !aligned16(v->data) || !aligned16(out->data))
    return fail(FIA_ERR_ALIGNMENT, "query/key/value/attention_out must be 16-byte aligned");
  if (g.layout == L_TND) {
    g.T1 = g.S1;
    g.T2 = g.S2;
    std::vector<int32_t> qs, ql, ks, kl;
    st = resolve_tnd(p->actual_seq_qlen, p->n_actual_seq_qlen, g.T1, qs, ql, "actual_seq_qlen");
    if (st != FIA_OK) return st;
    if (g.paged) {
      // the cache is paged, not TND: one key count per sequence
      if (Bk != int64_t(ql.size())) return fail(FIA_ERR_BLOCK_TABLE, "block_table must have one row per sequence");
      g.T2 = 0;
      st = resolve_lengths(p->actual_seq_kvlen, p->n_actual_seq_kvlen, Bk, g.S2, kl, "actual_seq_kvlen");
      ks.assign(kl.size(), 0);
    } else {
      st = resolve_tnd(p->actual_seq_kvlen, p->n_actual_seq_kvlen, g.T2, ks, kl, "actual_seq_kvlen");
    }
    if (st != FIA_OK) return st;
    if (ql.size() != kl.size()) return fail(FIA_ERR_SEQLEN, "TND lists must have the same number of entries");
    g.B = int64_t(ql.size());
    g.batches.resize(ql.size());
    for (size_t b = 0; b < ql.size(); ++b) g.batches[b] = BatchInfo{qs[b], ql[b], ks[b], kl[b]};
  } else {
    if (Bq != Bk) return fail(FIA_ERR_SHAPE, "query B=%lld, key B=%lld", (long long)Bq, (long long)Bk);
    g.B = Bq;
    g.T1 = g.T2 = 0;
    if (bsa && ((p->actual_seq_qlen == nullptr) != (p->actual_seq_kvlen == nullptr)))
      return fail(FIA_ERR_SEQLEN, "actual_seq_qlen and actual_seq_kvlen must be given together");
    std::vector<int32_t> ql, kl;
    st = resolve_lengths(p->actual_seq_qlen, p->n_actual_seq_qlen, g.B, g.S1, ql, "actual_seq_qlen");
    if (st != FIA_OK) return st;
    st = resolve_lengths(p->actual_seq_kvlen, p->n_actual_seq_kvlen, g.B, g.S2, kl, "actual_seq_kvlen");
    if (st != FIA_OK) return st;
    g.batches.resize(size_t(g.B));
    for (int64_t b = 0; b < g.B; ++b) g.batches[size_t(b)] = BatchInfo{0, ql[size_t(b)], 0, kl[size_t(b)]};
  }
  if (g.paged) {
    int64_t need_blocks = 0, max_blocks = 0;
    for (const auto& bi : g.batches) {
      need_blocks += (bi.kv_len + g.bs - 1) / g.bs;
      max_blocks = std::max<int64_t>(max_blocks, (bi.kv_len + g.bs - 1) / g.bs);
    }
    if (g.table_stride < max_blocks)
      return fail(FIA_ERR_BLOCK_TABLE, "block_table has fewer columns than maxBlocksPerSeq");
    if (g.nblk < need_blocks)
      return fail(FIA_ERR_BLOCK_TABLE, "blocknum %lld below the %lld blocks the lengths need", (long long)g.nblk,
                  (long long)need_blocks);
  }
  return FIA_OK;
}

// KV tiles that the 128 query rows from q0 visit under a causal mask.
int causal_tiles(const BatchInfo& bi, int q0, int mode) {
  const int off = mode == 3 ? bi.kv_len - bi.q_len : 0;
  const int last_row = std::min(q0 + kTileM - 1, bi.q_len - 1);
  const int maxkey = std::min(bi.kv_len - 1, last_row + off);
  return maxkey >= 0 ? maxkey / kTileN + 1 : 0;
}

// sparse_mode 4 (shift: d = kv_len - q_len) and the explicit mask's band (d =
// 0): K/V tiles that the rows [q0, q0 + 256) of a pair (both tiles walk the
// union of their bands) may see.
int band_tiles(const BatchInfo& bi, int q0, int pre, int next, bool shift) {
  const int64_t d = shift ? int64_t(bi.kv_len) - bi.q_len : 0;
  const int64_t last = std::min<int64_t>(q0 + 2 * kTileM - 1, bi.q_len - 1);
  const int64_t lo = std::max<int64_t>(0, q0 + d - pre);
  const int64_t hi = std::min<int64_t>(bi.kv_len - 1, last + d + next);
  return hi < lo ? 0 : int(hi / kTileN - lo / kTileN + 1);
}

// Work items: 256-row pairs of query tiles for the dense/causal kernel, single
// 128-row tiles for the block-sparse one.  cost = tile products (Q K^T + P V
// per 128 x 128 tile) the CTA runs.
void build_items(const Geometry& g, int prefill_mode, int causal_mode, std::vector<WorkItem>& items) {
  items.clear();
  const int rows = prefill_mode == kBlockSparse ? kTileM : 2 * kTileM;
  for (int64_t b = 0; b < g.B; ++b) {
    const BatchInfo& bi = g.batches[size_t(b)];
    const int nqt = (bi.q_len + rows - 1) / rows;
    const int full = (bi.kv_len + kTileN - 1) / kTileN;
    for (int64_t h = 0; h < g.N1; ++h)
      for (int qt = 0; qt < nqt; ++qt) {
        int cost = full;
        if (prefill_mode == kBand || prefill_mode == kMask) {
          const int q0 = qt * rows;
          const int n = band_tiles(bi, q0, g.band_pre, g.band_next, prefill_mode == kBand);
          cost = q0 + kTileM >= bi.q_len ? n : 2 * n;
        } else if (prefill_mode != kBlockSparse) {
          const int q0 = qt * rows;
          const int na = prefill_mode == kCausal ? causal_tiles(bi, q0, causal_mode) : full;
          const int nb = q0 + kTileM >= bi.q_len ? 0
                         : std::max(na, prefill_mode == kCausal ? causal_tiles(bi, q0 + kTileM, causal_mode) : full);
          cost = na + nb;
        }
        items.push_back(WorkItem{int32_t(b), int32_t(h), qt, cost});
      }
  }
  // Longest first (an LPT order for the hardware block scheduler); ties keep
  // the heads of one GQA group next to each other for L2 reuse of K/V.
  // When the keys and values the call reads are well beyond what L2 holds
  // (MHA, long sequences), the items of one (batch, kv head) run back to back
  // instead, so the CTAs reading the same K/V tiles are resident together:
  // units by total cost, longest first, and LPT inside a unit.
  double kv_bytes = 0.0;
  for (const auto& bi : g.batches) kv_bytes += double(bi.kv_len) * double(g.N2) * double(g.Dqk + g.Dv) * 2.0;
  constexpr double kL2Share = 48.0 * 1024 * 1024;   // about a third of the 126 MB L2
  if (prefill_mode != kBlockSparse && kv_bytes > kL2Share) {
    const int64_t group = g.N1 / g.N2;
    std::vector<int64_t> unit_cost(size_t(g.B * g.N2), 0);
    auto unit = [&](const WorkItem& w) { return int64_t(w.b) * g.N2 + w.h / group; };
    for (const auto& w : items) unit_cost[size_t(unit(w))] += w.cost;
    std::stable_sort(items.begin(), items.end(), [&](const WorkItem& a, const WorkItem& b) {
      const int64_t ua = unit(a), ub = unit(b);
      if (ua != ub) {
        const int64_t ca = unit_cost[size_t(ua)], cb = unit_cost[size_t(ub)];
        return ca != cb ? ca > cb : ua < ub;
      }
      return a.cost > b.cost;
    });
    return;
  }
  std::stable_sort(items.begin(), items.end(), [](const WorkItem& a, const WorkItem& b) { return a.cost > b.cost; });
}

size_t prefill_ws_bytes(size_t n_batches, size_t n_items) {
  return kHeader + align_up(n_batches * sizeof(BatchInfo), 256) + align_up(n_items * sizeof(WorkItem), 256);
}

// Tile codes of an explicit mask (one byte per 128 x 128 tile of each mask
// slice), kept in the workspace after the plan.
size_t mask_tiles_bytes(const Geometry& g) {
  if (g.mask == nullptr) return 0;
  const size_t n_mb = g.mask_sb > 0 ? size_t(g.B) : 1;
  return align_up(n_mb * size_t((g.mask_s1 + kTileM - 1) / kTileM) * size_t((g.mask_ss + kTileN - 1) / kTileN), 256);
}

size_t count_items(const Geometry& g) {
  size_t n = 0;
  for (const auto& bi : g.batches) n += size_t((bi.q_len + kTileM - 1) / kTileM) * size_t(g.N1);
  return n;
}

fia_status check_ws(void* ws, size_t have, size_t need) {
  if (ws == nullptr) return fail(FIA_ERR_WORKSPACE, "workspace is NULL");
  if (have < need) return fail(FIA_ERR_WORKSPACE, "workspace %zu bytes < required %zu", have, need);
  if (!aligned16(ws)) return fail(FIA_ERR_ALIGNMENT, "workspace not 16-byte aligned");
  return FIA_OK;
}

// Encode the (D, S, N, B) maps of a dense tensor (TND: (D, T, N, 1)).
fia_status dense_map(CUtensorMap* m, const fia_tensor* t, Layout L, int64_t B, int64_t N, int64_t S, int64_t D,
                     bool u8 = false) {
  uint64_t dims[4], st[3];
  const uint64_t e = u8 ? 1 : 2;
  if (L == L_BNSD) {
    dims[0] = D; dims[1] = S; dims[2] = N; dims[3] = B;
    st[0] = D * e; st[1] = S * D * e; st[2] = N * S * D * e;
  } else if (L == L_TND) {
    dims[0] = D; dims[1] = S; dims[2] = N; dims[3] = 1;
    st[0] = N * D * e; st[1] = D * e; st[2] = S * N * D * e;
  } else {
    dims[0] = D; dims[1] = S; dims[2] = N; dims[3] = B;
    st[0] = N * D * e; st[1] = D * e; st[2] = S * N * D * e;
  }
  return make_map(m, t->data, 4, dims, st, 128, u8);
}

// Launch the prefill (dense/causal) or block-sparse kernels for a validated geometry.
fia_status run_prefill(const Geometry& g, int mode, int causal_mode, const fia_tensor* q, const fia_tensor* k,
                       const fia_tensor* v, const fia_tensor* out, const fia_tensor* lse_t, const fia_params* prm,
                       const uint8_t* bsa_mask, int nqb, int nkb, int bx, int by, void* ws, size_t ws_bytes,
                       cudaStream_t stream) {
  std::vector<WorkItem> items;
  build_items(g, mode, causal_mode, items);
  const size_t plan_bytes = prefill_ws_bytes(g.batches.size(), items.size());
  // FP8: the value tensor converted to f16 once per call, after the plan;
  // an explicit mask's tile codes, after the plan
  const size_t need = plan_bytes + (g.fp8 ? align_up(size_t(numel(v)) * 2, 256) : 0) + mask_tiles_bytes(g);
  fia_status st = check_ws(ws, ws_bytes, need);
  if (st != FIA_OK) return st;
  float* lse = (prm->softmax_lse_flag && present(lse_t)) ? static_cast<float*>(lse_t->data) : nullptr;
  uint8_t* base = static_cast<uint8_t*>(ws);
  if (g.B == 0) return clear_status(base, stream);

  int64_t os[3], ls[3] = {0, 0, 0};
  bns_strides(g.layout, g.N1, g.S1, g.Dv, os);
  if (g.layout == L_TND) { ls[0] = 0; ls[1] = 1; ls[2] = g.N1; }
  else { ls[0] = g.N1 * g.S1; ls[1] = g.S1; ls[2] = 1; }

  // upload the plan
  std::vector<uint8_t> plan(plan_bytes - kHeader, 0);
  const size_t off_items = align_up(g.batches.size() * sizeof(BatchInfo), 256);
  memcpy(plan.data(), g.batches.data(), g.batches.size() * sizeof(BatchInfo));
  if (!items.empty()) memcpy(plan.data() + off_items, items.data(), items.size() * sizeof(WorkItem));
  st = cuda_check(cudaMemcpyAsync(base + kHeader, plan.data(), plan.size(), cudaMemcpyHostToDevice, stream), "plan upload");
  if (st != FIA_OK) return st;
  const BatchInfo* d_batches = reinterpret_cast<const BatchInfo*>(base + kHeader);
  const WorkItem* d_items = reinterpret_cast<const WorkItem*>(base + kHeader + off_items);

  // rows that no CTA writes: padding rows of the padded layouts
  if (g.layout != L_TND) {
    bool padded = false;
    for (const auto& bi : g.batches) padded |= bi.q_len < g.S1;
    if (padded) {
      const int64_t dims[4] = {g.B, g.N1, g.S1, g.Dv};
      st = cuda_check(launch_fill_rows(out->data, true, lse, dims, os, ls, d_batches, 0, stream), "fill rows");
      if (st != FIA_OK) return st;
    }
  }
  if (items.empty()) return clear_status(base, stream);
  if (g.S2 == 0 || (g.paged && g.nblk == 0)) {
    st = clear_status(base, stream);
    if (st != FIA_OK) return st;
    // K/V with S2 = 0 (or an empty pool, so every length is 0): every query
    // row is empty (out = 0, lse = +inf).
    const int64_t dims[4] = {g.layout == L_TND ? 1 : g.B, g.N1, g.layout == L_TND ? g.T1 : g.S1, g.Dv};
    int64_t os2[3] = {os[0], os[1], os[2]}, ls2[3] = {ls[0], ls[1], ls[2]};
    return cuda_check(launch_fill_rows(out->data, true, lse, dims, os2, ls2, d_batches, 1, stream), "fill rows");
  }

  PrefillParams pp;
  memset(&pp, 0, sizeof(pp));
  const int64_t Bmap = g.layout == L_TND ? 1 : g.B;
  st = dense_map(&pp.tm_q, q, g.layout, Bmap, g.N1, g.S1, g.D, g.fp8);
  if (st != FIA_OK) return st;
  if (g.paged) {
    // the pool as a (D, block_size, KV_N, blocknum) tensor: BNSD-like for
    // (blocknum, KV_N, bs, D), BSND-like for (blocknum, bs, KV_N*D)
    const Layout pl = g.kv_bnbd ? L_BNSD : L_BSND;
    st = dense_map(&pp.tm_k, k, pl, g.nblk, g.N2, g.bs, g.D);
    if (st != FIA_OK) return st;
    st = dense_map(&pp.tm_v, v, pl, g.nblk, g.N2, g.bs, g.D);
    if (st != FIA_OK) return st;
    pp.block_table = g.table;
    pp.table_stride = g.table_stride;
    pp.block_size = int(g.bs);
  } else if (g.fp8) {
    st = dense_map(&pp.tm_k, k, g.layout, Bmap, g.N2, g.S2, g.D, true);
    if (st != FIA_OK) return st;
    // V as f16 (2^-8 of each e4m3 value) in the workspace, same layout
    fia_tensor v16 = *v;
    v16.data = base + plan_bytes;
    v16.dtype = FIA_DTYPE_F16;
    st = cuda_check(launch_e4m3_to_f16(v->data, v16.data, numel(v), sm_count(), stream), "value conversion");
    if (st != FIA_OK) return st;
    st = dense_map(&pp.tm_v, &v16, g.layout, Bmap, g.N2, g.S2, g.Dv);
    if (st != FIA_OK) return st;
  } else {
    st = dense_map(&pp.tm_k, k, g.layout, Bmap, g.N2, g.S2, g.D);
    if (st != FIA_OK) return st;
    st = dense_map(&pp.tm_v, v, g.layout, Bmap, g.N2, g.S2, g.Dv);
    if (st != FIA_OK) return st;
  }
  // the score columns past 128 (MLA prefill): separate rope tensors, or
  // columns 128..191 of query / key
  pp.tm_qr = pp.tm_q;
  pp.tm_kr = pp.tm_k;
  pp.rope_col = 128;
  if (g.qr != nullptr) {
    st = dense_map(&pp.tm_qr, g.qr, g.layout, Bmap, g.N1, g.S1, 64);
    if (st != FIA_OK) return st;
    st = dense_map(&pp.tm_kr, g.kr, g.layout, Bmap, g.N2, g.S2, 64);
    if (st != FIA_OK) return st;
    pp.rope_col = 0;
  }
  pp.out = out->data;
  pp.lse = lse;
  pp.out_sb = os[0]; pp.out_sn = os[1]; pp.out_ss = os[2];
  pp.lse_sb = ls[0]; pp.lse_sn = ls[1]; pp.lse_ss = ls[2];
  pp.batches = d_batches;
  pp.items = d_items;
  pp.n_items = int(items.size());
  pp.prefetch_stride = sm_count();
  pp.num_heads = int(g.N1);
  pp.num_kv_heads = int(g.N2);
  pp.group = int(g.N1 / g.N2);
  pp.is_tnd = g.layout == L_TND;
  pp.causal_offset_mode = causal_mode;
  pp.band_pre = g.band_pre;
  pp.band_next = g.band_next;
  pp.attn_mask = g.mask;
  pp.mask_sb = g.mask_sb;
  pp.mask_ss = g.mask_ss;
  pp.mask_cs = g.mask_cs;
  if (mode == kMask) {
    // the tile codes, on the stream before the prefill kernel
    uint8_t* codes = base + plan_bytes + (g.fp8 ? align_up(size_t(numel(v)) * 2, 256) : 0);
    const int n_mb = g.mask_sb > 0 ? int(g.B) : 1;
    st = cuda_check(launch_mask_tile_summary(g.mask, g.mask_s1, g.mask_ss, n_mb, g.mask_cs, codes, stream),
                    "mask tile summary");
    if (st != FIA_OK) return st;
    pp.mask_tiles = codes;
    pp.mask_nkt = int((g.mask_ss + kTileN - 1) / kTileN);
    pp.mask_tiles_sb = g.mask_sb > 0 ? int64_t((g.mask_s1 + kTileM - 1) / kTileM) * pp.mask_nkt : 0;
  }
  pp.scale_log2 = float(prm->scale_value * 1.4426950408889634);
  pp.bsa_mask = bsa_mask;
  pp.bsa_nqb = nqb; pp.bsa_nkb = nkb; pp.bsa_x = bx; pp.bsa_y = by;
  pp.fp8_qscale = g.fp8_q;
  pp.fp8_kscale = g.fp8_k;
  pp.fp8_vscale = g.fp8_v;
  pp.fp8_nqs = g.fp8_nqs;
  pp.fp8_nks = g.fp8_nks;
  pp.status = make_status(base);
  return cuda_check(profiled(stream,
                             [&] {
                               if (g.fp8) return launch_bsa_fp8(pp, stream);
                               return mode == kBlockSparse ? launch_prefill(pp, int(g.D), g.bf16, mode, stream)
                                                           : launch_prefill_pair(pp, int(g.Dqk), int(g.Dv), g.bf16,
                                                                                 mode, stream);
                             }),
                    "prefill launch");
}

// An explicit atten_mask for the prefill kernels: bool / int8 / uint8, nonzero
// = masked, shapes (S1,S2), (B,S1,S2), (1,S1,S2), (B,1,S1,S2), (1,1,S1,S2)
// (npu_fused_infer_attention_score_v2 and npu_prompt_flash_attention,
// atten_mask).  Indices are batch-local (row i, key j of the batch); the last
// two dims must cover every batch's query and key lengths.
fia_status explicit_mask(const fia_tensor* mask, Geometry& g) {
  if (mask->dtype != FIA_DTYPE_BOOL && mask->dtype != FIA_DTYPE_U8 && mask->dtype != FIA_DTYPE_I8)
    return fail(FIA_ERR_DTYPE, "atten_mask must be bool, int8 or uint8");
  const int n = mask->ndim;
  if (n < 2 || n > 4) return fail(FIA_ERR_SHAPE, "atten_mask must be 2-D, 3-D or 4-D");
  const int64_t ms1 = mask->shape[n - 2], ms2 = mask->shape[n - 1];
  const int64_t mb = n >= 3 ? mask->shape[0] : 1;
  if (n == 4 && mask->shape[1] != 1) return fail(FIA_ERR_SHAPE, "4-D atten_mask must be (B or 1, 1, S1, S2)");
  if (mb != 1 && mb != g.B)
    return fail(FIA_ERR_SHAPE, "atten_mask batch dim %lld is neither 1 nor B=%lld", (long long)mb, (long long)g.B);
  int64_t maxq = 0, maxk = 0;
  for (const auto& bi : g.batches) { maxq = std::max<int64_t>(maxq, bi.q_len); maxk = std::max<int64_t>(maxk, bi.kv_len); }
  if (ms1 < maxq || ms2 < maxk)
    return fail(FIA_ERR_SHAPE, "atten_mask (%lld, %lld) smaller than the query / key lengths (%lld, %lld)",
                (long long)ms1, (long long)ms2, (long long)maxq, (long long)maxk);
  if (ms1 * ms2 > 0 && mask->data == nullptr) return fail(FIA_ERR_NULL, "atten_mask data is NULL");
  g.mask = static_cast<const uint8_t*>(mask->data);
  g.mask_ss = ms2;
  g.mask_s1 = ms1;
  g.mask_sb = mb > 1 ? ms1 * ms2 : 0;
  const uintptr_t a = reinterpret_cast<uintptr_t>(mask->data);
  g.mask_cs = 1;
  for (int cs : {16, 8, 4})
    if (a % cs == 0 && ms2 % cs == 0) { g.mask_cs = cs; break; }
  return FIA_OK;
}

// Mask semantics accepted by the prefill kernels.
fia_status prefill_mask_mode(const fia_params* p, const fia_tensor* mask, Geometry& g, int& mode, int& causal_mode) {
  const int64_t sm = p->sparse_mode;
  if (sm < 0 || sm > 8) return fail(FIA_ERR_SPARSE_MODE, "sparse_mode %lld not in 0..4", (long long)sm);
  if (sm >= 5) return fail(FIA_ERR_SPARSE_MODE, "sparse_mode %lld (prefix/global/dilated/block_local) is not supported", (long long)sm);
  if (sm == 0 || sm == 1) {
    causal_mode = 0;
    if (!present(mask)) {
      if (sm == 1) return fail(FIA_ERR_SPARSE_MODE, "sparse_mode 1 needs atten_mask");
      mode = kDense;   // no mask: pre_tokens / next_tokens are ignored
      return FIA_OK;
    }
    fia_status st = explicit_mask(mask, g);
    if (st != FIA_OK) return st;
    // mode 0 keeps the band pre_tokens .. next_tokens around the diagonal;
    // mode 1 (allMask) is the mask alone
    if (sm == 1) g.band_pre = g.band_next = 1 << 30;
    mode = kMask;
    return FIA_OK;
  }
  if (present(mask)) {
    // The 2048 x 2048 lower-triangular mask the pages ask for in modes 2/3 is
    // only a compressed form of the pattern; the kernels derive it from indices.
    const int64_t n = mask->ndim;
    const bool ok = (n >= 2 && n <= 4 && mask->shape[n - 1] == 2048 && mask->shape[n - 2] == 2048 &&
                     (n < 3 || mask->shape[0] == 1) && (n < 4 || mask->shape[1] == 1));
    if (!ok) return fail(FIA_ERR_SPARSE_MODE, "sparse_mode %lld mask must be (2048,2048)", (long long)sm);
  }
  mode = sm == 4 ? kBand : kCausal;
  causal_mode = int(sm);
  return FIA_OK;
}

fia_status clear_status(void* ws, cudaStream_t stream) {
  return cuda_check(cudaMemsetAsync(ws, 0, 8, stream), "status reset");
}

}  // namespace

namespace fia {
void set_last_error(int status, const char* message) {
  fail(static_cast<fia_status>(status), "%s", message);
}
}  // namespace fia

// ======================================================================= ABI
extern "C" {

void fia_params_init(fia_params* p) {
  if (p == nullptr) return;
  memset(p, 0, sizeof(*p));
  p->num_heads = 1;
  p->num_key_value_heads = 0;
  p->scale_value = 1.0;
  p->input_layout = "BSH";
  p->sparse_mode = 0;
  p->pre_tokens = kInt32Max;
  p->next_tokens = kInt32Max;
}

const char* fia_status_string(fia_status s) {
  switch (s) {
    case FIA_OK: return "FIA_OK";
    case FIA_ERR_NULL: return "FIA_ERR_NULL: required pointer missing";
    case FIA_ERR_DTYPE: return "FIA_ERR_DTYPE: unsupported or mismatched element type";
    case FIA_ERR_SHAPE: return "FIA_ERR_SHAPE: inconsistent shapes";
    case FIA_ERR_LAYOUT: return "FIA_ERR_LAYOUT: unknown input_layout";
    case FIA_ERR_UNSUPPORTED: return "FIA_ERR_UNSUPPORTED: not implemented by this library";
    case FIA_ERR_SEQLEN: return "FIA_ERR_SEQLEN: invalid actual_seq list";
    case FIA_ERR_BLOCK_TABLE: return "FIA_ERR_BLOCK_TABLE: invalid block_table / block_size";
    case FIA_ERR_WORKSPACE: return "FIA_ERR_WORKSPACE: workspace missing or too small";
    case FIA_ERR_CUDA: return "FIA_ERR_CUDA: CUDA call failed";
    case FIA_ERR_TIMEOUT: return "FIA_ERR_TIMEOUT: a bounded device wait ran out";
    case FIA_ERR_HEADS: return "FIA_ERR_HEADS: invalid num_heads / num_key_value_heads";
    case FIA_ERR_SPARSE_MODE: return "FIA_ERR_SPARSE_MODE: invalid sparse_mode or mask";
    case FIA_ERR_ALIGNMENT: return "FIA_ERR_ALIGNMENT: pointer not 16-byte aligned";
  }
  return "unknown fia_status";
}

const char* fia_last_error(void) { return g_last_error.c_str(); }

void fia_profile_next_call(void* start_event, void* stop_event) {
  g_prof_start = static_cast<cudaEvent_t>(start_event);
  g_prof_stop = static_cast<cudaEvent_t>(stop_event);
}

void fia_debug_set_wait_limit_ns(uint64_t ns) { g_wait_limit_ns.store(ns, std::memory_order_relaxed); }
void fia_debug_set_decode_path(int path) { g_decode_force_tc.store(path == 1 ? 1 : 0, std::memory_order_relaxed); }

fia_status fia_device_status(const void* workspace, void* stream) {
  if (workspace == nullptr) return fail(FIA_ERR_NULL, "workspace is NULL");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  fia_status st = cuda_check(cudaStreamSynchronize(s), "stream sync");
  if (st != FIA_OK) return st;
  unsigned long long word = 0;   // (epoch << 8) | code
  st = cuda_check(cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost), "status read");
  if (st != FIA_OK) return st;
  return static_cast<fia_status>(word & 0xffu);
}

// ---------------------------------------------------------------- prefill
fia_status fia_prefill_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                          const fia_tensor* atten_mask, const fia_params* params,
                                          const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                                          size_t* workspace_bytes) {
  return fia_prefill_paged_get_workspace_size(query, key, value, nullptr, atten_mask, params, attention_out,
                                              softmax_lse, workspace_bytes);
}

fia_status fia_prefill(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                       const fia_tensor* atten_mask, const fia_params* params, const fia_tensor* attention_out,
                       const fia_tensor* softmax_lse, void* workspace, size_t workspace_bytes, void* stream) {
  return fia_prefill_paged(query, key, value, nullptr, atten_mask, params, attention_out, softmax_lse, workspace,
                           workspace_bytes, stream);
}

// block_table NULL: contiguous key/value (fia_prefill).
fia_status fia_prefill_paged_get_workspace_size(const fia_tensor* query, const fia_tensor* key_cache,
                                                const fia_tensor* value_cache, const fia_tensor* block_table,
                                                const fia_tensor* atten_mask, const fia_params* params,
                                                const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                                                size_t* workspace_bytes) {
  if (workspace_bytes == nullptr) return fail(FIA_ERR_NULL, "workspace_bytes is NULL");
  *workspace_bytes = kHeader;
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;   // empty query
  Geometry g;
  fia_status st = prefill_geometry(query, key_cache, value_cache, params, attention_out, false, g, block_table);
  if (st != FIA_OK) return st;
  int mode, cm;
  st = prefill_mask_mode(params, atten_mask, g, mode, cm);
  if (st != FIA_OK) return st;
  st = check_lse(softmax_lse, params, g.layout, g.B, g.N1, g.S1, g.T1);
  if (st != FIA_OK) return st;
  *workspace_bytes = prefill_ws_bytes(g.batches.size(), count_items(g)) + mask_tiles_bytes(g);
  return FIA_OK;
}

fia_status fia_prefill_paged(const fia_tensor* query, const fia_tensor* key_cache, const fia_tensor* value_cache,
                             const fia_tensor* block_table, const fia_tensor* atten_mask, const fia_params* params,
                             const fia_tensor* attention_out, const fia_tensor* softmax_lse, void* workspace,
                             size_t workspace_bytes, void* stream) {
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;
  Geometry g;
  fia_status st = prefill_geometry(query, key_cache, value_cache, params, attention_out, false, g, block_table);
  if (st != FIA_OK) return st;
  int mode, cm;
  st = prefill_mask_mode(params, atten_mask, g, mode, cm);
  if (st != FIA_OK) return st;
  st = check_lse(softmax_lse, params, g.layout, g.B, g.N1, g.S1, g.T1);
  if (st != FIA_OK) return st;
  return run_prefill(g, mode, cm, query, key_cache, value_cache, attention_out, softmax_lse, params, nullptr, 0, 0, 0,
                     0, workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

fia_status fia_prefill_mla_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                              const fia_tensor* query_rope, const fia_tensor* key_rope,
                                              const fia_tensor* atten_mask, const fia_params* params,
                                              const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                                              size_t* workspace_bytes) {
  if (workspace_bytes == nullptr) return fail(FIA_ERR_NULL, "workspace_bytes is NULL");
  *workspace_bytes = kHeader;
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;   // empty query
  Geometry g;
  fia_status st = prefill_geometry(query, key, value, params, attention_out, false, g, nullptr, true, query_rope,
                                   key_rope);
  if (st != FIA_OK) return st;
  int mode, cm;
  st = prefill_mask_mode(params, atten_mask, g, mode, cm);
  if (st != FIA_OK) return st;
  st = check_lse(softmax_lse, params, g.layout, g.B, g.N1, g.S1, g.T1);
  if (st != FIA_OK) return st;
  *workspace_bytes = prefill_ws_bytes(g.batches.size(), count_items(g));
  return FIA_OK;
}

fia_status fia_prefill_mla(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                           const fia_tensor* query_rope, const fia_tensor* key_rope, const fia_tensor* atten_mask,
                           const fia_params* params, const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                           void* workspace, size_t workspace_bytes, void* stream) {
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;
  Geometry g;
  fia_status st = prefill_geometry(query, key, value, params, attention_out, false, g, nullptr, true, query_rope,
                                   key_rope);
  if (st != FIA_OK) return st;
  int mode, cm;
  st = prefill_mask_mode(params, atten_mask, g, mode, cm);
  if (st != FIA_OK) return st;
  st = check_lse(softmax_lse, params, g.layout, g.B, g.N1, g.S1, g.T1);
  if (st != FIA_OK) return st;
  return run_prefill(g, mode, cm, query, key, value, attention_out, softmax_lse, params, nullptr, 0, 0, 0, 0, workspace,
                     workspace_bytes, static_cast<cudaStream_t>(stream));
}

// ------------------------------------------------------------ block-sparse
// FP8 (q_scale non-NULL): e4m3 query / key / value with fp32 dequant scales
// (BSA "FP8特性说明"): q_scale (B, N1, ceil(maxQS / 128), 1), k_scale and
// v_scale (B, N2, ceil(maxKVS / Y), 1); block_shape X = 128, Y = 256 or 512.
static fia_status bsa_validate(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                               const fia_tensor* mask, const int64_t* block_shape, const fia_params* params,
                               const fia_tensor* out, const fia_tensor* lse, Geometry& g, int& nqb, int& nkb,
                               const fia_tensor* q_scale = nullptr, const fia_tensor* k_scale = nullptr,
                               const fia_tensor* v_scale = nullptr) {
  const bool fp8 = q_scale != nullptr || k_scale != nullptr || v_scale != nullptr;
  fia_status st = prefill_geometry(query, key, value, params, out, true, g, nullptr, false, nullptr, nullptr, fp8);
  if (st != FIA_OK) return st;
  if (block_shape == nullptr) return fail(FIA_ERR_NULL, "block_shape is required");
  const int64_t X = block_shape[0], Y = block_shape[1];
  if (X <= 0 || Y <= 0 || Y % 128 != 0) return fail(FIA_ERR_SHAPE, "block_shape [%lld,%lld]: X > 0 and Y a multiple of 128", (long long)X, (long long)Y);
  if (X % 128 != 0) return fail(FIA_ERR_UNSUPPORTED, "block_shape X=%lld: this library needs a multiple of 128", (long long)X);
  // FP8 without a mask: every block kept (dense FP8 attention)
  if (!present(mask) && !fp8) return fail(FIA_ERR_NULL, "block_sparse_mask is required");
  if (present(mask) && mask->dtype != FIA_DTYPE_U8 && mask->dtype != FIA_DTYPE_BOOL)
    return fail(FIA_ERR_DTYPE, "block_sparse_mask must be uint8/bool");
  int64_t maxq = 0, maxk = 0;
  for (const auto& bi : g.batches) { maxq = std::max<int64_t>(maxq, bi.q_len); maxk = std::max<int64_t>(maxk, bi.kv_len); }
  if (g.layout != L_TND && params->actual_seq_qlen == nullptr) { maxq = g.S1; maxk = g.S2; }
  nqb = int((maxq + X - 1) / X);
  nkb = int((maxk + Y - 1) / Y);
  if (present(mask) &&
      !(mask->ndim == 4 && mask->shape[0] == g.B && mask->shape[1] == g.N1 && mask->shape[2] == nqb && mask->shape[3] == nkb))
    return fail(FIA_ERR_SHAPE, "block_sparse_mask must be (B, N1, %d, %d)", nqb, nkb);
  if (params->sparse_mode != 0) return fail(FIA_ERR_SPARSE_MODE, "block-sparse attention takes no sparse_mode");
  if (fp8) {
    if (X != 128 || (Y != 256 && Y != 512))
      return fail(FIA_ERR_SHAPE, "FP8 block_shape must be [128, 256] or [128, 512] (the quantisation blocks)");
    const int64_t nqs = (maxq + 127) / 128, nks = (maxk + Y - 1) / Y;
    auto scale_ok = [&](const fia_tensor* t, int64_t heads, int64_t blocks) {
      return present(t) && t->dtype == FIA_DTYPE_F32 && t->ndim == 4 && t->shape[0] == g.B && t->shape[1] == heads &&
             t->shape[2] == blocks && t->shape[3] == 1 && reinterpret_cast<uintptr_t>(t->data) % 4 == 0;
    };
    if (!scale_ok(q_scale, g.N1, nqs))
      return fail(FIA_ERR_SHAPE, "q_dequant_scale must be fp32 (B, N1, %lld, 1)", (long long)nqs);
    if (!scale_ok(k_scale, g.N2, nks) || !scale_ok(v_scale, g.N2, nks))
      return fail(FIA_ERR_SHAPE, "k/v_dequant_scale must be fp32 (B, N2, %lld, 1)", (long long)nks);
    g.fp8_q = static_cast<const float*>(q_scale->data);
    g.fp8_k = static_cast<const float*>(k_scale->data);
    g.fp8_v = static_cast<const float*>(v_scale->data);
    g.fp8_nqs = int(nqs);
    g.fp8_nks = int(nks);
  }
  return check_lse(lse, params, g.layout, g.B, g.N1, g.S1, g.T1);
}

fia_status bsa_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                  const fia_tensor* block_sparse_mask, const int64_t* block_shape,
                                  const fia_params* params, const fia_tensor* attention_out,
                                  const fia_tensor* softmax_lse, size_t* workspace_bytes) {
  if (workspace_bytes == nullptr) return fail(FIA_ERR_NULL, "workspace_bytes is NULL");
  *workspace_bytes = kHeader;
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;
  Geometry g;
  int nqb = 0, nkb = 0;
  fia_status st = bsa_validate(query, key, value, block_sparse_mask, block_shape, params, attention_out, softmax_lse, g, nqb, nkb);
  if (st != FIA_OK) return st;
  *workspace_bytes = prefill_ws_bytes(g.batches.size(), count_items(g));
  return FIA_OK;
}

fia_status bsa_forward(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                       const fia_tensor* block_sparse_mask, const int64_t* block_shape, const fia_params* params,
                       const fia_tensor* attention_out, const fia_tensor* softmax_lse, void* workspace,
                       size_t workspace_bytes, void* stream) {
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;
  Geometry g;
  int nqb = 0, nkb = 0;
  fia_status st = bsa_validate(query, key, value, block_sparse_mask, block_shape, params, attention_out, softmax_lse, g, nqb, nkb);
  if (st != FIA_OK) return st;
  return run_prefill(g, kBlockSparse, 0, query, key, value, attention_out, softmax_lse, params,
                     static_cast<const uint8_t*>(block_sparse_mask->data), nqb, nkb, int(block_shape[0]),
                     int(block_shape[1]), workspace, workspace_bytes, static_cast<cudaStream_t>(stream));
}

fia_status bsa_fp8_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                      const fia_tensor* block_sparse_mask, const int64_t* block_shape,
                                      const fia_tensor* q_dequant_scale, const fia_tensor* k_dequant_scale,
                                      const fia_tensor* v_dequant_scale, const fia_params* params,
                                      const fia_tensor* attention_out, const fia_tensor* softmax_lse,
                                      size_t* workspace_bytes) {
  if (workspace_bytes == nullptr) return fail(FIA_ERR_NULL, "workspace_bytes is NULL");
  *workspace_bytes = kHeader;
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;
  if (q_dequant_scale == nullptr || k_dequant_scale == nullptr || v_dequant_scale == nullptr)
    return fail(FIA_ERR_NULL, "FP8 attention needs all three dequant scales");
  Geometry g;
  int nqb = 0, nkb = 0;
  fia_status st = bsa_validate(query, key, value, block_sparse_mask, block_shape, params, attention_out, softmax_lse,
                               g, nqb, nkb, q_dequant_scale, k_dequant_scale, v_dequant_scale);
  if (st != FIA_OK) return st;
  *workspace_bytes = prefill_ws_bytes(g.batches.size(), count_items(g)) + align_up(size_t(numel(value)) * 2, 256);
  return FIA_OK;
}

fia_status bsa_forward_fp8(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                           const fia_tensor* block_sparse_mask, const int64_t* block_shape,
                           const fia_tensor* q_dequant_scale, const fia_tensor* k_dequant_scale,
                           const fia_tensor* v_dequant_scale, const fia_params* params,
                           const fia_tensor* attention_out, const fia_tensor* softmax_lse, void* workspace,
                           size_t workspace_bytes, void* stream) {
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;
  if (q_dequant_scale == nullptr || k_dequant_scale == nullptr || v_dequant_scale == nullptr)
    return fail(FIA_ERR_NULL, "FP8 attention needs all three dequant scales");
  Geometry g;
  int nqb = 0, nkb = 0;
  fia_status st = bsa_validate(query, key, value, block_sparse_mask, block_shape, params, attention_out, softmax_lse,
                               g, nqb, nkb, q_dequant_scale, k_dequant_scale, v_dequant_scale);
  if (st != FIA_OK) return st;
  return run_prefill(g, kBlockSparse, 0, query, key, value, attention_out, softmax_lse, params,
                     present(block_sparse_mask) ? static_cast<const uint8_t*>(block_sparse_mask->data) : nullptr,
                     nqb, nkb, int(block_shape[0]), int(block_shape[1]), workspace, workspace_bytes,
                     static_cast<cudaStream_t>(stream));
}

}  // extern "C"

// ================================================================== decode
namespace {

struct DecodeGeometry {
  Layout layout;
  int64_t B, N1, N2, D, Dv;
  bool bf16, paged, mla, kv_bnbd;
  int64_t bs, nblk, S2;
  std::vector<int32_t> kv_len;
  int64_t q_sb, q_sn, q_ss, o_sb, o_sn, o_ss;
  int64_t QS = 1;         // query tokens per sequence
  int q_causal = 0;       // with QS > 1: sparse_mode 0, 2 or 3
  const uint8_t* key_mask = nullptr;   // atten_mask (Q_S = 1): one row of key bytes per batch
  int64_t key_mask_sb = 0;             // 0: one row for every batch
  int64_t rows() const { return (N1 / N2) * QS; }
};

fia_status decode_geometry(const fia_tensor* q, const fia_tensor* k, const fia_tensor* v, const fia_tensor* qr,
                           const fia_tensor* kr, const fia_tensor* table, const fia_tensor* mask, const fia_params* p,
                           const fia_tensor* out, DecodeGeometry& g) {
  if (p == nullptr) return fail(FIA_ERR_NULL, "params is NULL");
  if (!given(q) || !given(k) || !given(v) || !given(out))
    return fail(FIA_ERR_NULL, "query/key/value/attention_out required");
  g.layout = parse_layout(p->input_layout);
  if (g.layout == L_BAD) return fail(FIA_ERR_LAYOUT, "input_layout '%s' not supported", p->input_layout);
  if (g.layout == L_TND) return fail(FIA_ERR_UNSUPPORTED, "TND decode is not implemented");
  if (!is_half(q->dtype) || k->dtype != q->dtype || v->dtype != q->dtype || out->dtype != q->dtype)
    return fail(FIA_ERR_DTYPE, "query/key/value/attention_out must share fp16 or bf16");
  if (present(qr) != present(kr)) return fail(FIA_ERR_SHAPE, "query_rope and key_rope must be given together");
  g.mla = present(qr);
  fia_status st = resolve_heads(p, g.N1, g.N2, g.mla ? 128 : 64);
  if (st != FIA_OK) return st;
  if (!same_shape(q, out)) return fail(FIA_ERR_SHAPE, "attention_out must have the query's shape");
  int64_t Bq, Sq, D;
  st = dense_dims(q, g.layout, g.N1, Bq, Sq, D, "query");
  if (st != FIA_OK) return st;
  // Several new tokens per sequence: the unit's rows are its heads x tokens,
  // at most 64 (the widest kernel tile), and the mask over the Q_S x S_kv block
  // is none (0) or causal (2 top-left, 3 bottom-right).
  if (Sq < 1 || Sq > 16) return fail(FIA_ERR_UNSUPPORTED, "fia_decode takes Q_S in 1..16 (got %lld)", (long long)Sq);
  g.QS = Sq;
  if (Sq > 1) {
    const int64_t sm = p->sparse_mode;
    if (sm != 0 && sm != 2 && sm != 3)
      return fail(FIA_ERR_UNSUPPORTED, "decode with Q_S > 1 takes sparse_mode 0, 2 or 3 (got %lld)", (long long)sm);
    g.q_causal = int(sm);
  }
  g.B = Bq;
  g.D = D;
  g.bf16 = q->dtype == FIA_DTYPE_BF16;
  if (!(p->scale_value > 0.0) || !std::isfinite(p->scale_value))
    return fail(FIA_ERR_UNSUPPORTED, "scale_value must be finite and > 0");
  if (!aligned16(q->data) || !aligned16(k->data) || !aligned16(v->data) || !aligned16(out->data))
    return fail(FIA_ERR_ALIGNMENT, "query/key/value/attention_out must be 16-byte aligned");
  int64_t qs[3];
  bns_strides(g.layout, g.N1, Sq, D, qs);
  g.q_sb = qs[0]; g.q_sn = qs[1]; g.q_ss = qs[2];
  g.o_sb = qs[0]; g.o_sn = qs[1]; g.o_ss = qs[2];
  g.paged = present(table);
  if (g.paged) {
    if (table->dtype != FIA_DTYPE_I32 || table->ndim != 2 || table->shape[0] != g.B)
      return fail(FIA_ERR_BLOCK_TABLE, "block_table must be int32 (B, maxBlocksPerSeq)");
    if (!aligned16(table->data)) return fail(FIA_ERR_ALIGNMENT, "block_table not 16-byte aligned");
    if (p->actual_seq_kvlen == nullptr) return fail(FIA_ERR_SEQLEN, "page attention needs actual_seq_kvlen");
    g.bs = p->block_size;
    if (g.bs <= 0 || g.bs % 16 != 0 || !(128 % g.bs == 0 || g.bs % 128 == 0))
      return fail(FIA_ERR_BLOCK_TABLE, "block_size %lld: multiple of 16 dividing 128, or multiple of 128", (long long)g.bs);
    if (!same_shape(k, v)) return fail(FIA_ERR_SHAPE, "key and value shapes differ");
    if (k->ndim == 4) {
      g.kv_bnbd = true;
      if (k->shape[1] != g.N2 || k->shape[2] != g.bs || k->shape[3] != D)
        return fail(FIA_ERR_SHAPE, "paged key must be (blocknum, KV_N, block_size, D)");
    } else if (k->ndim == 3) {
      g.kv_bnbd = false;
      if (k->shape[1] != g.bs || k->shape[2] != g.N2 * D)
        return fail(FIA_ERR_SHAPE, "paged key must be (blocknum, block_size, KV_N*D)");
    } else {
      return fail(FIA_ERR_SHAPE, "paged key must be 3-D or 4-D");
    }
    g.nblk = k->shape[0];
    g.S2 = table->shape[1] * g.bs;
    st = resolve_lengths(p->actual_seq_kvlen, p->n_actual_seq_kvlen, g.B, g.S2, g.kv_len, "actual_seq_kvlen");
    if (st != FIA_OK) return st;
    int64_t need_blocks = 0, max_blocks = 0;
    for (auto L : g.kv_len) {
      need_blocks += (L + g.bs - 1) / g.bs;
      max_blocks = std::max<int64_t>(max_blocks, (L + g.bs - 1) / g.bs);
    }
    if (table->shape[1] < max_blocks) return fail(FIA_ERR_BLOCK_TABLE, "block_table has fewer columns than maxBlocksPerSeq");
    if (g.nblk < need_blocks && !g.mla) return fail(FIA_ERR_BLOCK_TABLE, "blocknum %lld below the %lld blocks the lengths need", (long long)g.nblk, (long long)need_blocks);
  } else {
    if (!same_shape(k, v)) return fail(FIA_ERR_SHAPE, "key and value shapes differ");
    int64_t Bk, Dk;
    st = dense_dims(k, g.layout, g.N2, Bk, g.S2, Dk, "key");
    if (st != FIA_OK) return st;
    if (Bk != g.B || Dk != D) return fail(FIA_ERR_SHAPE, "key must be (B, ..., D) like the query");
    st = resolve_lengths(p->actual_seq_kvlen, p->n_actual_seq_kvlen, g.B, g.S2, g.kv_len, "actual_seq_kvlen");
    if (st != FIA_OK) return st;
    g.bs = 0;
  }
  if (g.mla) {
    // MLA: key = value = the 512-d latent cache, plus a 64-d rope part of q and k
    if (present(mask)) return fail(FIA_ERR_UNSUPPORTED, "atten_mask with MLA decode is not implemented");
    if (D != 512) return fail(FIA_ERR_UNSUPPORTED, "MLA decode takes a 512-d latent query (got %lld)", (long long)D);
    if (g.QS != 1) return fail(FIA_ERR_UNSUPPORTED, "MLA decode takes Q_S = 1");
    if (g.N2 != 1) return fail(FIA_ERR_UNSUPPORTED, "MLA decode takes num_key_value_heads = 1");
    if (g.N1 > 128) return fail(FIA_ERR_UNSUPPORTED, "MLA decode takes at most 128 query heads");
    if (qr->dtype != q->dtype || kr->dtype != q->dtype) return fail(FIA_ERR_DTYPE, "query_rope/key_rope must match query");
    if (qr->ndim != q->ndim || numel(qr) != numel(q) / 8 || qr->shape[qr->ndim - 1] != 64)
      return fail(FIA_ERR_SHAPE, "query_rope must be the query's shape with last dim 64");
    if (kr->ndim != k->ndim || numel(kr) != numel(k) / 8 || kr->shape[kr->ndim - 1] != 64)
      return fail(FIA_ERR_SHAPE, "key_rope must be the key's shape with last dim 64");
    if (!aligned16(qr->data) || !aligned16(kr->data)) return fail(FIA_ERR_ALIGNMENT, "rope tensors not 16-byte aligned");
    if (k->data != v->data) return fail(FIA_ERR_UNSUPPORTED, "MLA decode takes value = key (the latent cache)");
    g.Dv = 512;
    return FIA_OK;
  }
  if (D != 64 && D != 128) return fail(FIA_ERR_UNSUPPORTED, "decode head dim %lld (kernels take 64 or 128)", (long long)D);
  if (g.rows() > 64)
    return fail(FIA_ERR_UNSUPPORTED, "decode rows per KV head (Q_N / KV_N x Q_S = %lld) above 64", (long long)g.rows());
  g.Dv = D;
  if (present(mask)) {
    // the incremental case's atten_mask (npu_fused_infer_attention_score_v2,
    // atten_mask with Q_S = 1): (B, KV_S), (B, 1, KV_S) or (B, 1, 1, KV_S),
    // batch dim 1 broadcast; nonzero bytes mask their key
    if (g.QS != 1) return fail(FIA_ERR_UNSUPPORTED, "decode atten_mask is taken with Q_S = 1 only");
    if (mask->dtype != FIA_DTYPE_BOOL && mask->dtype != FIA_DTYPE_U8 && mask->dtype != FIA_DTYPE_I8)
      return fail(FIA_ERR_DTYPE, "atten_mask must be bool, int8 or uint8");
    const int n = mask->ndim;
    if (n < 2 || n > 4) return fail(FIA_ERR_SHAPE, "decode atten_mask must be (B, KV_S), (B, 1, KV_S) or (B, 1, 1, KV_S)");
    for (int i = 1; i < n - 1; ++i)
      if (mask->shape[i] != 1)
        return fail(FIA_ERR_SHAPE, "decode atten_mask must be (B, KV_S), (B, 1, KV_S) or (B, 1, 1, KV_S)");
    const int64_t mb = mask->shape[0], ms = mask->shape[n - 1];
    if (mb != 1 && mb != g.B)
      return fail(FIA_ERR_SHAPE, "atten_mask batch dim %lld is neither 1 nor B=%lld", (long long)mb, (long long)g.B);
    int64_t maxk = 0;
    for (auto L : g.kv_len) maxk = std::max<int64_t>(maxk, L);
    if (ms < maxk)
      return fail(FIA_ERR_SHAPE, "atten_mask has %lld keys, below the longest sequence (%lld)", (long long)ms,
                  (long long)maxk);
    if (mb * ms > 0 && mask->data == nullptr) return fail(FIA_ERR_NULL, "atten_mask data is NULL");
    g.key_mask = static_cast<const uint8_t*>(mask->data);
    g.key_mask_sb = mb > 1 ? ms : 0;
  }
  return FIA_OK;
}

// Copies of the group's head rows in the decode kernel's 128-row query tile.

struct DecodePlan {
  std::vector<DecodeSeg> segs;
  std::vector<int32_t> cta_seg;
  std::vector<int2> unit_parts;
  int n_cta = 0, n_units = 0;
};

// How many stages ahead the decode producers warm L2 (0: off).
int g_decode_l2_ahead = 0;

// Charge, in stages, for every unit piece (segment) a CTA runs: the end of a
// segment drains the pipeline, sums and writes the partials, and a split
// unit costs a merge at the end of the CTA that finishes it last.  Tuned on
// the paged GQA decode kernel at B=16, U[1,4096] (same-box sweep, us per call
// back to back): 1 -> 26.1, 2 -> 25.3, 3 -> 24.9, 4 -> 24.6, 5 -> 25.0,
// 7 -> 25.6; the 4-token decode has its optimum between 3 and 5.
constexpr double kDecodeSegmentCost = 4.0;
// MLA decode (32-token stages; same-box sweep at B=32, L=8192, ms per call:
// 1 -> 0.2470, 3 -> 0.2458, 8 -> 0.2495).
constexpr double kMlaSegmentCost = 3.0;

// Deals the stages of all units (unit order = batch-major, then kv head) to at
// most n_sm CTAs so that every CTA carries about the same cost: one per stage
// plus seg_cost per segment.  Greedy fill against a capacity that grows
// until the stages fit the CTAs.  Within a CTA, the pieces of units that other
// CTAs share go first: the CTA that completes a unit merges it, and a split
// unit finished early is merged while the CTA still streams, not at its end.
void plan_decode(const DecodeGeometry& g, int n_sm, DecodePlan& pl, int stage_keys, double seg_cost) {
  pl.n_units = int(g.B * g.N2);
  std::vector<int32_t> nst(size_t(pl.n_units));
  int64_t T = 0, nonempty = 0;
  for (int u = 0; u < pl.n_units; ++u) {
    nst[size_t(u)] = int32_t((g.kv_len[size_t(u / g.N2)] + stage_keys - 1) / stage_keys);
    T += nst[size_t(u)];
    nonempty += nst[size_t(u)] > 0;
  }
  pl.unit_parts.assign(size_t(pl.n_units), int2{0, 0});
  pl.segs.clear();
  const int max_cta = int(std::min<int64_t>(std::min<int64_t>(n_sm, kMaxDecodeCtas), T));
  if (max_cta == 0) {
    pl.n_cta = 0;
    pl.cta_seg.assign(1, 0);
    return;
  }
  double cap = (double(T) + seg_cost * double(nonempty + max_cta - 1)) / max_cta;
  for (int attempt = 0; attempt < 1000; ++attempt, cap *= 1.005) {
    pl.segs.clear();
    pl.cta_seg.assign(1, 0);
    int c = 0;
    double acc = 0.0;
    bool fits = true;
    for (int u = 0; u < pl.n_units && fits; ++u) {
      int begin = 0, left = nst[size_t(u)];
      pl.unit_parts[size_t(u)] = int2{int(pl.segs.size()), 0};
      while (left > 0) {
        if (acc > 0.0 && acc + seg_cost + 1.0 > cap) {
          pl.cta_seg.push_back(int32_t(pl.segs.size()));
          if (++c >= max_cta) { fits = false; break; }
          acc = 0.0;
        }
        acc += seg_cost;
        const int room = std::max(1, int(cap - acc));
        const int k = std::min(left, room);
        pl.segs.push_back(DecodeSeg{u, begin, begin + k, int32_t(pl.segs.size())});
        pl.unit_parts[size_t(u)].y += 1;
        acc += k;
        begin += k;
        left -= k;
      }
    }
    if (fits) {
      pl.cta_seg.push_back(int32_t(pl.segs.size()));
      pl.n_cta = int(pl.cta_seg.size()) - 1;
      for (int c = 0; c < pl.n_cta; ++c)
        std::stable_partition(pl.segs.begin() + pl.cta_seg[size_t(c)], pl.segs.begin() + pl.cta_seg[size_t(c) + 1],
                              [&](const DecodeSeg& sg) { return pl.unit_parts[size_t(sg.unit)].y > 1; });
      return;
    }
  }
  // unreachable in practice: one CTA per stage always fits
  pl.n_cta = 0;
  pl.cta_seg.assign(1, 0);
}

struct DecodeWsLayout {
  size_t off_ctr, off_plan, off_po, off_pl, total;
};

// 32-bit plan words of a plan: cta_seg, segments (4 words), unit parts (2
// words), kv lengths (1 word).
size_t decode_plan_words(size_t n_segs, size_t n_cta, size_t n_units, size_t B) {
  return align_up(n_cta + 1, 4) + 4 * n_segs + 2 * n_units + B + 2;
}

// Workspace: status word | per-unit counters | plan (used when it does not
// fit in the kernel parameters) | partial O | partial lse.
DecodeWsLayout decode_ws_layout(size_t n_segs, size_t n_cta, size_t n_units, size_t B, size_t rows, size_t D) {
  DecodeWsLayout w;
  size_t o = kHeader;
  w.off_ctr = o; o += align_up(n_units * sizeof(unsigned long long), 256);
  w.off_plan = o; o += align_up(decode_plan_words(n_segs, n_cta, n_units, B) * sizeof(int32_t), 256);
  w.off_po = o; o += align_up(n_segs * rows * D * sizeof(float), 256);
  w.off_pl = o; o += align_up(n_segs * rows * sizeof(float), 256);
  w.total = o;
  return w;
}

// Upper bound over every plan the call can make (at most kMaxDecodeCtas CTAs,
// so at most n_units + kMaxDecodeCtas segments).
size_t decode_ws_bound(const DecodeGeometry& g) {
  const size_t n_units = size_t(g.B * g.N2);
  const size_t n_segs = n_units + kMaxDecodeCtas;
  const size_t rows = size_t(g.rows());
  return decode_ws_layout(n_segs, kMaxDecodeCtas, n_units, size_t(g.B), rows, size_t(g.D)).total;
}

// The decode plan as words (layout in internal.h): 16-bit words into the
// kernel parameters when every value and the whole plan fit, else 32-bit
// words for the workspace.  Returns true for the inline form.
bool pack_decode_plan(const DecodePlan& pl, const std::vector<int32_t>& kv_len, DecodeParams& dp,
                      std::vector<int32_t>& wide) {
  const size_t n_cta = size_t(pl.n_cta), n_segs = pl.segs.size(), n_units = pl.unit_parts.size(), B = kv_len.size();
  const int seg = int(align_up(n_cta + 1, 4));
  const int unit = seg + int(4 * n_segs);
  const int len = int(align_up(size_t(unit) + 2 * n_units, 2));
  dp.plan_seg = seg;
  dp.plan_unit = unit;
  dp.plan_len = len;
  bool fits = size_t(len) + 2 * B <= size_t(kDecodePlanInline) && n_segs <= 32767 && n_units <= 32767;
  for (size_t i = 0; fits && i < n_segs; ++i) fits = pl.segs[i].stage_end <= 32767;
  if (fits) {
    int16_t* w = dp.plan_inline;
    memset(w, 0, sizeof(dp.plan_inline));
    for (size_t c = 0; c <= n_cta; ++c) w[c] = int16_t(pl.cta_seg[c]);
    for (size_t i = 0; i < n_segs; ++i) {
      const DecodeSeg& sg = pl.segs[i];
      w[seg + 4 * i] = int16_t(sg.unit);
      w[seg + 4 * i + 1] = int16_t(sg.stage_begin);
      w[seg + 4 * i + 2] = int16_t(sg.stage_end);
      w[seg + 4 * i + 3] = int16_t(sg.part);
    }
    for (size_t u = 0; u < n_units; ++u) {
      w[unit + 2 * u] = int16_t(pl.unit_parts[u].x);
      w[unit + 2 * u + 1] = int16_t(pl.unit_parts[u].y);
    }
    for (size_t b = 0; b < B; ++b) {
      const uint32_t L = uint32_t(kv_len[b]);
      w[len + 2 * b] = int16_t(uint16_t(L & 0xffffu));
      w[len + 2 * b + 1] = int16_t(uint16_t(L >> 16));
    }
    return true;
  }
  wide.assign(size_t(len) + B, 0);
  for (size_t c = 0; c <= n_cta; ++c) wide[c] = pl.cta_seg[c];
  for (size_t i = 0; i < n_segs; ++i) {
    const DecodeSeg& sg = pl.segs[i];
    wide[seg + 4 * i] = sg.unit;
    wide[seg + 4 * i + 1] = sg.stage_begin;
    wide[seg + 4 * i + 2] = sg.stage_end;
    wide[seg + 4 * i + 3] = sg.part;
  }
  for (size_t u = 0; u < n_units; ++u) {
    wide[unit + 2 * u] = pl.unit_parts[u].x;
    wide[unit + 2 * u + 1] = pl.unit_parts[u].y;
  }
  for (size_t b = 0; b < B; ++b) wide[len + b] = kv_len[b];
  return false;
}

// MLA: stages of 32 keys, one plan slot per CTA pair, partials per output half.
constexpr int kMlaStageKeys = 32;
constexpr int kMlaMaxPairs = 128;

struct MlaWsLayout {
  size_t off_ctr, off_segs, off_cta, off_units, off_len, off_po, off_pl, total;
};

MlaWsLayout mla_ws_layout(size_t n_segs, size_t n_pairs, size_t B, size_t N1, bool plan_in_ws) {
  MlaWsLayout w;
  size_t o = kHeader;
  w.off_ctr = o; o += align_up(2 * B * sizeof(unsigned long long), 256);
  w.off_segs = o; o += plan_in_ws ? align_up(n_segs * sizeof(DecodeSeg), 256) : 0;
  w.off_cta = o; o += plan_in_ws ? align_up((n_pairs + 1) * sizeof(int32_t), 256) : 0;
  w.off_units = o; o += plan_in_ws ? align_up(B * sizeof(int2), 256) : 0;
  w.off_len = o; o += plan_in_ws ? align_up(B * sizeof(int32_t), 256) : 0;
  w.off_po = o; o += align_up(2 * n_segs * N1 * 256 * sizeof(float), 256);
  w.off_pl = o; o += align_up(2 * n_segs * N1 * sizeof(float), 256);
  w.total = o;
  return w;
}

size_t mla_ws_bound(const DecodeGeometry& g) {
  const size_t n_segs = size_t(g.B) + kMlaMaxPairs;
  return mla_ws_layout(n_segs, kMlaMaxPairs, size_t(g.B), size_t(g.N1), true).total;
}

fia_status check_decode_lse(const fia_tensor* lse, const fia_params* p, int64_t B, int64_t N1, int64_t QS) {
  if (p->softmax_lse_flag == 0) return FIA_OK;
  if (!present(lse)) return fail(FIA_ERR_NULL, "softmax_lse_flag set but softmax_lse absent");
  if (lse->dtype != FIA_DTYPE_F32) return fail(FIA_ERR_DTYPE, "softmax_lse must be fp32");
  if (!(lse->ndim == 4 && lse->shape[0] == B && lse->shape[1] == N1 && lse->shape[2] == QS && lse->shape[3] == 1))
    return fail(FIA_ERR_SHAPE, "softmax_lse must be (B, N1, Q_S, 1)");
  return FIA_OK;
}

// Copies a decode plan into the workspace (one host-to-device copy on the
// call's stream; the staging buffer may go once the call returns).
fia_status upload_plan(const DecodePlan& pl, const std::vector<int32_t>& kv_len, uint8_t* base, size_t off_segs,
                       size_t off_cta, size_t off_units, size_t off_len, size_t off_end, cudaStream_t stream) {
  std::vector<uint8_t> plan(off_end - off_segs, 0);
  memcpy(plan.data(), pl.segs.data(), pl.segs.size() * sizeof(DecodeSeg));
  memcpy(plan.data() + (off_cta - off_segs), pl.cta_seg.data(), pl.cta_seg.size() * sizeof(int32_t));
  memcpy(plan.data() + (off_units - off_segs), pl.unit_parts.data(), pl.unit_parts.size() * sizeof(int2));
  memcpy(plan.data() + (off_len - off_segs), kv_len.data(), kv_len.size() * sizeof(int32_t));
  return cuda_check(cudaMemcpyAsync(base + off_segs, plan.data(), plan.size(), cudaMemcpyHostToDevice, stream),
                    "plan upload");
}

// MLA decode (key = value = the latent cache, plus rope): plan the batches'
// 32-key stages over CTA pairs and launch the pair kernel.
fia_status run_mla(const DecodeGeometry& g, const fia_tensor* query, const fia_tensor* key, const fia_tensor* qr,
                   const fia_tensor* kr, const fia_tensor* block_table, const fia_params* params,
                   const fia_tensor* attention_out, const fia_tensor* softmax_lse, void* workspace,
                   size_t workspace_bytes, cudaStream_t stream) {
  DecodePlan pl;
  const int pairs = std::max(1, std::min(kMlaMaxPairs, sm_count() / 2));
  plan_decode(g, pairs, pl, kMlaStageKeys, kMlaSegmentCost);
  const MlaWsLayout w = mla_ws_layout(pl.segs.size(), size_t(pl.n_cta), size_t(g.B), size_t(g.N1), true);
  fia_status st = check_ws(workspace, workspace_bytes, w.total);
  if (st != FIA_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(workspace);
  MlaParams mp;
  memset(&mp, 0, sizeof(mp));
  st = upload_plan(pl, g.kv_len, base, w.off_segs, w.off_cta, w.off_units, w.off_len, w.off_po, stream);
  if (st != FIA_OK) return st;
  mp.segs = reinterpret_cast<const DecodeSeg*>(base + w.off_segs);
  mp.cta_seg = reinterpret_cast<const int32_t*>(base + w.off_cta);
  mp.unit_parts = reinterpret_cast<const int2*>(base + w.off_units);
  mp.kv_len = reinterpret_cast<const int32_t*>(base + w.off_len);
  const uint64_t qrows = uint64_t(g.B * g.N1);
  uint64_t dims[2], strides[1];
  dims[0] = 512; dims[1] = qrows; strides[0] = 1024;
  st = make_map(&mp.tm_q, query->data, 2, dims, strides, 128);
  if (st != FIA_OK) return st;
  dims[0] = 64; strides[0] = 128;
  st = make_map(&mp.tm_qr, qr->data, 2, dims, strides, 128);
  if (st != FIA_OK) return st;
  if (pl.n_cta > 0) {
    const uint64_t rows = uint64_t(g.paged ? g.nblk * g.bs : g.B * g.S2);
    mp.box_rows = g.paged ? int(std::min<int64_t>(g.bs, 32)) : 32;
    mp.block_size = g.paged ? int(g.bs) : (1 << 30);
    mp.row_per_blk = g.paged ? g.bs : g.S2;
    mp.block_table = g.paged ? static_cast<const int32_t*>(block_table->data) : nullptr;
    mp.table_stride = g.paged ? block_table->shape[1] : 0;
    dims[0] = 512; dims[1] = rows; strides[0] = 1024;
    st = make_map(&mp.tm_lat, key->data, 2, dims, strides, uint32_t(mp.box_rows));
    if (st != FIA_OK) return st;
    dims[0] = 64; strides[0] = 128;
    st = make_map(&mp.tm_rope, kr->data, 2, dims, strides, uint32_t(mp.box_rows));
    if (st != FIA_OK) return st;
  }
  mp.out = attention_out->data;
  mp.out_sb = g.o_sb;
  mp.out_sn = g.o_sn;
  mp.lse = (params->softmax_lse_flag && present(softmax_lse)) ? static_cast<float*>(softmax_lse->data) : nullptr;
  mp.lse_sb = g.N1;
  mp.lse_sn = 1;
  mp.part_o = reinterpret_cast<float*>(base + w.off_po);
  mp.part_lse = reinterpret_cast<float*>(base + w.off_pl);
  mp.part_stride_o = int64_t(pl.segs.size()) * g.N1 * 256;
  mp.part_stride_lse = int64_t(pl.segs.size()) * g.N1;
  mp.unit_counter = reinterpret_cast<unsigned long long*>(base + w.off_ctr);
  mp.n_pairs = pl.n_cta;
  mp.n_units = pl.n_units;
  mp.num_heads = int(g.N1);
  mp.scale_log2 = float(params->scale_value * 1.4426950408889634);
  mp.status = make_status(base);
  return cuda_check(profiled(stream, [&] { return launch_mla(mp, g.bf16, stream); }), "MLA decode launch");
}

}  // namespace

extern "C" {

fia_status fia_decode_get_workspace_size(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                                         const fia_tensor* query_rope, const fia_tensor* key_rope,
                                         const fia_tensor* block_table, const fia_tensor* atten_mask,
                                         const fia_params* params, const fia_tensor* attention_out,
                                         const fia_tensor* softmax_lse, size_t* workspace_bytes) {
  if (workspace_bytes == nullptr) return fail(FIA_ERR_NULL, "workspace_bytes is NULL");
  *workspace_bytes = kHeader;
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;
  DecodeGeometry g;
  fia_status st = decode_geometry(query, key, value, query_rope, key_rope, block_table, atten_mask, params, attention_out, g);
  if (st != FIA_OK) return st;
  st = check_decode_lse(softmax_lse, params, g.B, g.N1, g.QS);
  if (st != FIA_OK) return st;
  *workspace_bytes = g.mla ? mla_ws_bound(g) : decode_ws_bound(g);
  return FIA_OK;
}

fia_status fia_decode(const fia_tensor* query, const fia_tensor* key, const fia_tensor* value,
                      const fia_tensor* query_rope, const fia_tensor* key_rope, const fia_tensor* block_table,
                      const fia_tensor* atten_mask, const fia_params* params, const fia_tensor* attention_out,
                      const fia_tensor* softmax_lse, void* workspace, size_t workspace_bytes, void* stream) {
  if (query != nullptr && query->ndim > 0 && numel(query) == 0) return FIA_OK;
  DecodeGeometry g;
  fia_status st = decode_geometry(query, key, value, query_rope, key_rope, block_table, atten_mask, params, attention_out, g);
  if (st != FIA_OK) return st;
  st = check_decode_lse(softmax_lse, params, g.B, g.N1, g.QS);
  if (st != FIA_OK) return st;
  cudaStream_t stream_t = static_cast<cudaStream_t>(stream);
  if (g.mla)
    return run_mla(g, query, key, query_rope, key_rope, block_table, params, attention_out, softmax_lse, workspace,
                   workspace_bytes, stream_t);
  DecodePlan pl;
  plan_decode(g, sm_count(), pl, 128, kDecodeSegmentCost);
  const size_t rows = size_t(g.rows());
  const DecodeWsLayout w = decode_ws_layout(pl.segs.size(), size_t(pl.n_cta), size_t(pl.n_units), size_t(g.B), rows,
                                            size_t(g.D));
  st = check_ws(workspace, workspace_bytes, w.total);
  if (st != FIA_OK) return st;
  uint8_t* base = static_cast<uint8_t*>(workspace);

  // DecodeParams carries a 6 KB plan area: kept off the stack
  thread_local DecodeParams dp;
  memset(&dp, 0, offsetof(DecodeParams, plan_inline));
  thread_local std::vector<int32_t> wide;
  if (!pack_decode_plan(pl, g.kv_len, dp, wide)) {
    st = cuda_check(cudaMemcpyAsync(base + w.off_plan, wide.data(), wide.size() * sizeof(int32_t),
                                    cudaMemcpyHostToDevice, stream_t),
                    "plan upload");
    if (st != FIA_OK) return st;
    dp.plan_ws = reinterpret_cast<const int32_t*>(base + w.off_plan);
  }
  if (!pl.segs.empty()) {
    uint64_t dims[2], strides[1];
    if (g.paged) {
      if (g.kv_bnbd) {
        dims[0] = uint64_t(g.D); dims[1] = uint64_t(g.nblk * g.N2 * g.bs);
        dp.row_per_blk = g.N2 * g.bs; dp.row_per_head = g.bs; dp.col_per_head = 0;
      } else {
        dims[0] = uint64_t(g.N2 * g.D); dims[1] = uint64_t(g.nblk * g.bs);
        dp.row_per_blk = g.bs; dp.row_per_head = 0; dp.col_per_head = int32_t(g.D);
      }
      dp.block_size = int(g.bs);
      dp.box_rows = int(std::min<int64_t>(g.bs, 128));
      dp.block_table = static_cast<const int32_t*>(block_table->data);
      dp.table_stride = block_table->shape[1];
    } else {
      if (g.layout == L_BNSD) {
        dims[0] = uint64_t(g.D); dims[1] = uint64_t(g.B * g.N2 * g.S2);
        dp.row_per_blk = g.N2 * g.S2; dp.row_per_head = g.S2; dp.col_per_head = 0;
      } else {
        dims[0] = uint64_t(g.N2 * g.D); dims[1] = uint64_t(g.B * g.S2);
        dp.row_per_blk = g.S2; dp.row_per_head = 0; dp.col_per_head = int32_t(g.D);
      }
      dp.block_size = 1 << 30;
      dp.box_rows = 128;
      dp.block_table = nullptr;
    }
    strides[0] = dims[0] * 2;
    st = make_map(&dp.tm_k, key->data, 2, dims, strides, uint32_t(dp.box_rows));
    if (st != FIA_OK) return st;
    st = make_map(&dp.tm_v, value->data, 2, dims, strides, uint32_t(dp.box_rows));
    if (st != FIA_OK) return st;
  }
  dp.q = query->data;
  dp.q_sb = g.q_sb; dp.q_sn = g.q_sn; dp.q_ss = g.q_ss;
  dp.out = attention_out->data;
  dp.out_sb = g.o_sb; dp.out_sn = g.o_sn; dp.out_ss = g.o_ss;
  dp.lse = (params->softmax_lse_flag && present(softmax_lse)) ? static_cast<float*>(softmax_lse->data) : nullptr;
  dp.lse_sb = g.N1 * g.QS; dp.lse_sn = g.QS; dp.lse_ss = 1;   // (B, N1, Q_S, 1)
  dp.q_tokens = int(g.QS);
  dp.q_causal = g.q_causal;
  dp.key_mask = g.key_mask;
  dp.key_mask_sb = g.key_mask_sb;
  dp.rows = int(g.rows());
  dp.part_o = reinterpret_cast<float*>(base + w.off_po);
  dp.part_lse = reinterpret_cast<float*>(base + w.off_pl);
  dp.unit_counter = reinterpret_cast<unsigned long long*>(base + w.off_ctr);
  dp.n_cta = pl.n_cta;
  dp.n_units = pl.n_units;
  dp.batch = int(g.B);
  dp.num_heads = int(g.N1);
  dp.num_kv_heads = int(g.N2);
  dp.group = int(g.N1 / g.N2);
  dp.scale_log2 = float(params->scale_value * 1.4426950408889634);
  dp.l2_ahead = g_decode_l2_ahead;
  dp.force_tc = g_decode_force_tc.load(std::memory_order_relaxed);
  dp.status = make_status(base);
  return cuda_check(profiled(stream_t, [&] { return launch_decode(dp, int(g.D), g.bf16, stream_t); }),
                    "decode launch");
}


fia_status fia_debug_plan_decode(const int32_t* kv_len, int B, int N2, int n_cta_max, int32_t* cta_seg,
                                 int cta_seg_cap, int32_t* segs, int segs_cap, int32_t* unit_parts,
                                 int unit_parts_cap, int* n_cta, int* n_segs) {
  if (kv_len == nullptr || cta_seg == nullptr || segs == nullptr || unit_parts == nullptr || n_cta == nullptr ||
      n_segs == nullptr)
    return fail(FIA_ERR_NULL, "fia_debug_plan_decode: NULL argument");
  if (B < 0 || N2 < 1 || n_cta_max < 1) return fail(FIA_ERR_SHAPE, "fia_debug_plan_decode: B >= 0, N2 >= 1, CTAs >= 1");
  DecodeGeometry g;
  g.B = B;
  g.N2 = N2;
  g.kv_len.assign(kv_len, kv_len + B);
  DecodePlan pl;
  plan_decode(g, n_cta_max, pl, 128, kDecodeSegmentCost);
  if (int64_t(pl.n_cta) + 1 > cta_seg_cap || int64_t(pl.segs.size()) * 4 > segs_cap ||
      int64_t(pl.n_units) * 2 > unit_parts_cap)
    return fail(FIA_ERR_SHAPE, "fia_debug_plan_decode: output capacity too small");
  for (int c = 0; c <= pl.n_cta; ++c) cta_seg[c] = pl.n_cta > 0 ? pl.cta_seg[size_t(c)] : 0;
  for (size_t i = 0; i < pl.segs.size(); ++i) {
    segs[4 * i] = pl.segs[i].unit;
    segs[4 * i + 1] = pl.segs[i].stage_begin;
    segs[4 * i + 2] = pl.segs[i].stage_end;
    segs[4 * i + 3] = pl.segs[i].part;
  }
  for (int u = 0; u < pl.n_units; ++u) {
    unit_parts[2 * u] = pl.unit_parts[size_t(u)].x;
    unit_parts[2 * u + 1] = pl.unit_parts[size_t(u)].y;
  }
  *n_cta = pl.n_cta;
  *n_segs = int(pl.segs.size());
  return FIA_OK;
}

}  // extern "C"

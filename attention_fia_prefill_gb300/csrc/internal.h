// Launch-side structures shared by the host API (fia_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <atomic>
#include <cstdint>

#include "ptx.cuh"

namespace fia {

// Raises a kernel's dynamic shared-memory limit on the first launch on each
// device; later launches skip the driver call (it costs microseconds of host
// time on every launch otherwise).
template <auto Kernel>
cudaError_t set_smem_once(int bytes) {
  static std::atomic<unsigned long long> done{0};   // one bit per device
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
  if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
  return e;
}

constexpr int kTileM = 128;   // query rows per prefill CTA
constexpr int kTileN = 128;   // keys per KV tile

// Per-batch geometry after length resolution.  For TND, q_start/kv_start are
// the first token row of the batch; for the padded layouts they are 0.
struct BatchInfo {
  int32_t q_start, q_len, kv_start, kv_len;
};

// One prefill CTA of (batch b, query head h): query rows [q_tile*128,
// q_tile*128+128) for the block-sparse kernel, [q_tile*256, q_tile*256+256)
// (two 128-row tiles) for the dense/causal kernel.
struct WorkItem {
  int32_t b, h, q_tile, cost;
};

// kBand: sparse_mode 4, key j of query row i allowed when
// i + d - pre <= j <= i + d + next, d = kv_len - q_len of the batch.
// kMask: an explicit atten_mask (sparse_mode 0 with a mask, 1), key j of row i
// allowed when mask[i][j] == 0 and i - pre <= j <= i + next (mode 1: no band).
enum PrefillMode : int { kDense = 0, kCausal = 1, kBlockSparse = 2, kBand = 3, kMask = 4 };

struct PrefillParams {
  // 4-D maps (D, S, N, B); TND uses (D, T, N, 1).  With a paged cache the K/V
  // maps cover the pool as (D, block_size, KV_N, blocknum).
  CUtensorMap tm_q, tm_k, tm_v;
  // scores over 192 columns (MLA prefill): columns 128..191 of Q / K come from
  // tm_qr / tm_kr at column rope_col (separate 64-wide rope tensors, rope_col
  // 0, or the same 192-wide tensors, rope_col 128)
  CUtensorMap tm_qr, tm_kr;
  int rope_col;
  void* out;                      // attention_out, query layout, element type of q
  float* lse;                     // nullable
  int64_t out_sb, out_sn, out_ss; // element strides of out for (b, n, s)
  int64_t lse_sb, lse_sn, lse_ss; // element strides of lse
  const BatchInfo* batches;
  const WorkItem* items;
  int n_items;
  int prefetch_stride;            // pair kernel: item blockIdx.x + stride gets its Q warmed in L2 (0: off)
  int num_heads, num_kv_heads, group;
  int is_tnd;
  int causal_offset_mode;         // 2: diagonal j <= i; 3: j <= i + kv_len - q_len
  int band_pre, band_next;        // kBand / kMask: pre_tokens / next_tokens, clamped to +-2^30
  const uint8_t* attn_mask;       // kMask: byte (i, j) of batch b at b * mask_sb + i * mask_ss + j
  int64_t mask_sb, mask_ss;       // mask_sb = 0 for a mask shared by all batches
  int mask_cs;                    // copy granule in bytes (16, 8, 4: alignment of base and rows; 1: plain loads)
  // explicit mask: one code per 128 x 128 tile of the mask (0 no key masked,
  // 1 some, 2 every one), [mask batches][mask_nqt][mask_nkt]; a batch's codes
  // at b * mask_tiles_sb (0 for a mask shared by all batches)
  const uint8_t* mask_tiles;
  int mask_nkt;
  int64_t mask_tiles_sb;
  const int32_t* block_table;     // paged K/V: [B, table_stride] block ids; nullptr = contiguous K/V
  int64_t table_stride;
  int block_size;                 // a multiple of 128: a 128-key tile lies in one block
  float scale_log2;               // scale * log2(e)
  const uint8_t* bsa_mask;        // [B, N1, nqb, nkb]
  int bsa_nqb, bsa_nkb, bsa_x, bsa_y;
  // FP8 block-sparse: dequant scales [B, N1, fp8_nqs] (128 query rows per
  // block) and [B, N2, fp8_nks] (bsa_y key rows per block) for K and V
  const float* fp8_qscale;
  const float* fp8_kscale;
  const float* fp8_vscale;
  int fp8_nqs, fp8_nks;
  DevStatus status;
};

// Paged / contiguous decode.  A unit is (batch, kv head).  Every unit's keys
// are cut into 128-token stages; the stages of all units, in unit order, are
// dealt out to the CTAs (one per SM), so a CTA may end one unit and start the
// next: each such piece is a "segment", and each segment leaves one partial
// (O / l, lse) per query row of the unit.
struct DecodeSeg {
  int32_t unit, stage_begin, stage_end, part;   // part = global segment index
};

// The plan travels in the kernel parameters when it fits (16-bit words, so
// the launch needs no host-to-device copy and can overlap the previous kernel);
// larger plans are copied into the workspace as 32-bit words.  Word layout:
// cta_seg[n_cta + 1] at 0, segments (unit, stage_begin, stage_end, part) at
// plan_seg, unit parts (first segment, count) at plan_unit, kv lengths at
// plan_len (inline: low / high 16-bit halves; workspace: one word each).
constexpr int kDecodePlanInline = 3072;   // 16-bit words (6 KB)

struct DecodeParams {
  CUtensorMap tm_k, tm_v;         // 2-D maps (row width in elements, rows), box (64, box_rows)
  int box_rows;                   // min(block_size, 128)
  int block_size;                 // tokens per page (contiguous caches: a whole sequence)
  int64_t row_per_blk;            // map row of token 0 of block id 1 (paged) / of batch 1 (contiguous)
  int64_t row_per_head;           // map row offset between kv heads
  int32_t col_per_head;           // map column offset between kv heads
  const int32_t* block_table;     // nullable (contiguous)
  int64_t table_stride;
  // Row r of a unit (rows = group * q_tokens): head kvh * group + r / q_tokens,
  // query token r % q_tokens.  Element strides of q / out / lse for (b, n, s).
  const void* q;
  int64_t q_sb, q_sn, q_ss;
  void* out;
  int64_t out_sb, out_sn, out_ss;
  float* lse;                     // nullable
  int64_t lse_sb, lse_sn, lse_ss;
  int q_tokens;                   // Q_S (1..16)
  int q_causal;                   // with Q_S > 1: 0 none, 2 key <= token, 3 key <= S_kv - Q_S + token
  const uint8_t* key_mask;        // nullable: atten_mask of Q_S = 1, byte j of batch b at b * key_mask_sb + j
  int64_t key_mask_sb;            // (nonzero: key j masked); 0 broadcasts one row to every batch
  int rows;                       // group * q_tokens (<= 64)
  float* part_o;                  // [n_segments, rows, D]
  float* part_lse;                // [n_segments, rows] natural log, -inf = empty
  unsigned long long* unit_counter;   // [n_units] (unit_tag(epoch): high half) | segments finished
  int n_cta, n_units;
  int batch, num_heads, num_kv_heads, group;
  float scale_log2;
  int l2_ahead;                   // producers warm L2 with the tiles of the stage this many ahead (0: off)
  int force_tc;                   // 1: the tcgen05 kernel even for units of <= 16 rows (tests)
  DevStatus status;
  const int32_t* plan_ws;         // the plan in the workspace (32-bit words), or nullptr: plan_inline
  int plan_seg, plan_unit, plan_len;
  alignas(16) int16_t plan_inline[kDecodePlanInline];
};

// MLA decode (latent D = 512 shared by key and value, plus a 64-d rope part of
// the key).  A unit is a batch; the plan's segments are run by CTA pairs:
// CTA 2c + h computes the scores of pair c's segments over all query heads and
// accumulates half h of the 512-wide output.
struct MlaParams {
  CUtensorMap tm_lat, tm_rope;    // 2-D maps over the cache: (512 | 64 columns, rows), box (64, box_rows)
  CUtensorMap tm_q, tm_qr;        // 2-D maps over q (512 columns) and q_rope (64), rows = b * Q_N + h, box (64, 128)
  int box_rows;                   // min(block_size, 32)
  int block_size;
  int64_t row_per_blk;            // cache row of token 0 of block 1 (paged) / of batch 1 (contiguous)
  const int32_t* block_table;     // nullable (contiguous)
  int64_t table_stride;
  void* out;                      // attention_out (B, 1, Q_N, 512)
  int64_t out_sb, out_sn;
  float* lse;                     // nullable, (B, Q_N, 1, 1)
  int64_t lse_sb, lse_sn;
  float* part_o;                  // [2 halves][n_segments][Q_N][256]
  float* part_lse;                // [2 halves][n_segments][Q_N]
  int64_t part_stride_o, part_stride_lse;   // elements per half
  unsigned long long* unit_counter;   // [B][2] (unit_tag(epoch): high half) | segments finished
  int n_pairs, n_units;
  int num_heads;
  float scale_log2;
  DevStatus status;
  const DecodeSeg* segs;
  const int32_t* cta_seg;         // per pair
  const int2* unit_parts;
  const int32_t* kv_len;
};

// Records the detail string fia_last_error() returns on this thread.
void set_last_error(int status, const char* message);

// Host-side launchers (defined next to their kernels).
cudaError_t launch_prefill(const PrefillParams& p, int head_dim, bool bf16, int mode, cudaStream_t s);
cudaError_t launch_prefill_pair(const PrefillParams& p, int head_dim_qk, int head_dim_v, bool bf16, int mode,
                                cudaStream_t s);
cudaError_t launch_bsa_fp8(const PrefillParams& p, cudaStream_t s);
// Tile codes of an explicit atten_mask (PrefillParams::mask_tiles): mask
// [n_mb][s1][s2] bytes (n_mb slices s1 * s2 apart), codes [n_mb][nqt][nkt].
cudaError_t launch_mask_tile_summary(const uint8_t* mask, int64_t s1, int64_t s2, int n_mb, int cs, uint8_t* codes,
                                     cudaStream_t s);
// e4m3 bytes -> f16 holding 2^-8 of each value (the FP8 path's value tensor);
// n_bytes a multiple of 16, both pointers 16-byte aligned.
cudaError_t launch_e4m3_to_f16(const void* src, void* dst, int64_t n_bytes, int n_sm, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, int head_dim, bool bf16, cudaStream_t s);
cudaError_t launch_mla(const MlaParams& p, bool bf16, cudaStream_t s);
cudaError_t launch_fill_rows(void* out, bool half_type, float* lse, const int64_t* dims, const int64_t* out_strides,
                             const int64_t* lse_strides, const BatchInfo* batches, int mode, cudaStream_t s);

}  // namespace fia

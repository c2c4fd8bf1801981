// Launch-side structures shared by the host API (fia_api.cu) and the kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace fia {

constexpr int kTileM = 128;   // query rows per prefill CTA
constexpr int kTileN = 128;   // keys per KV tile

// Per-batch geometry after length resolution.  For TND, q_start/kv_start are
// the first token row of the batch; for the padded layouts they are 0.
struct BatchInfo {
  int32_t q_start, q_len, kv_start, kv_len;
};

// One prefill CTA: query rows [q_tile*128, q_tile*128+128) of (batch b, query head h).
struct WorkItem {
  int32_t b, h, q_tile, cost;
};

enum PrefillMode : int { kDense = 0, kCausal = 1, kBlockSparse = 2 };

struct PrefillParams {
  CUtensorMap tm_q, tm_k, tm_v;   // 4-D maps (D, S, N, B); TND uses (D, T, N, 1)
  void* out;                      // attention_out, query layout, element type of q
  float* lse;                     // nullable
  int64_t out_sb, out_sn, out_ss; // element strides of out for (b, n, s)
  int64_t lse_sb, lse_sn, lse_ss; // element strides of lse
  const BatchInfo* batches;
  const WorkItem* items;
  int n_items;
  int num_heads, num_kv_heads, group;
  int is_tnd;
  int causal_offset_mode;         // 2: diagonal j <= i; 3: j <= i + kv_len - q_len
  float scale_log2;               // scale * log2(e)
  const uint8_t* bsa_mask;        // [B, N1, nqb, nkb]
  int bsa_nqb, bsa_nkb, bsa_x, bsa_y;
  uint32_t* status;
};

// Paged / contiguous decode (Q_S = 1).  The KV sequence of every unit
// (batch, kv head, head block) is cut into 128-token stages; the stages of all
// units, in unit order, are dealt out evenly to the CTAs (one per SM), so a CTA
// may finish one unit and start the next ("segments").  Each segment leaves one
// partial (O / l, lse) that the combine kernel merges.
struct DecodeSeg {
  int32_t unit, stage_begin, stage_end, part;
};

struct DecodeParams {
  CUtensorMap tm_k, tm_v;         // 2-D maps (row width in elements, rows), box (64, box_rows)
  int box_rows;                   // min(block_size, 128)
  int block_size;                 // tokens per page (contiguous caches: a whole sequence)
  int64_t row_per_blk;            // map row of token 0 of block id 1 (paged) / of batch 1 (contiguous)
  int64_t row_per_head;           // map row offset between kv heads
  int32_t col_per_head;           // map column offset between kv heads
  const int32_t* block_table;     // nullable (contiguous)
  int64_t table_stride;
  const void* q;                  // element (b, h, d) at q[b*q_sb + h*q_sn + d]
  int64_t q_sb, q_sn;
  const int32_t* kv_len;          // [B] on device
  void* out;
  int64_t out_sb, out_sn;
  float* lse;                     // nullable
  int64_t lse_sb, lse_sn;
  float* part_o;                  // [n_parts, G, D]
  float* part_lse;                // [n_parts, G] natural log, -inf = empty
  const DecodeSeg* segs;
  const int32_t* cta_seg;         // [n_cta + 1]
  const int2* unit_parts;         // [n_units] {first part, n parts}
  int n_cta, n_units;
  int batch, num_heads, num_kv_heads, group, heads_per_unit, head_blocks;
  float scale_log2;
  uint32_t* status;
};

struct MLAParams {
  const void* q;                  // (b, h, 512) via strides
  const void* q_rope;             // (b, h, 64)
  int64_t q_sb, q_sn, qr_sb, qr_sn;
  const void* latent;             // (nblk, bs, 512)
  const void* rope;               // (nblk, bs, 64)
  const int32_t* block_table;
  int64_t table_stride;
  int block_size;
  const int32_t* kv_len;          // [B]
  void* out;                      // (b, h, 512)
  int64_t out_sb, out_sn;
  float* lse;
  int64_t lse_sb, lse_sn;
  float* part_o;                  // [n_parts, 128, 512]
  float* part_lse;                // [n_parts, 128]
  const int4* chunks;             // {b, first page, n pages, part index}
  const int2* unit_parts;         // per b: {first part, n parts}
  int n_chunks;
  int num_heads;
  float scale_log2;
  uint32_t* status;
};

// Records the detail string fia_last_error() returns on this thread.
void set_last_error(int status, const char* message);

// Host-side launchers (defined next to their kernels).
cudaError_t launch_prefill(const PrefillParams& p, int head_dim, bool bf16, int mode, cudaStream_t s);
cudaError_t launch_decode(const DecodeParams& p, int head_dim, bool bf16, int part, cudaStream_t s);
cudaError_t launch_mla_decode(const MLAParams& p, int n_batches, cudaStream_t s);
cudaError_t launch_fill_rows(void* out, bool half_type, float* lse, const int64_t* dims, const int64_t* out_strides,
                             const int64_t* lse_strides, const BatchInfo* batches, int mode, cudaStream_t s);

}  // namespace fia

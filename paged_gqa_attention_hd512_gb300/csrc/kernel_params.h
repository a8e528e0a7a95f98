// kernel_params.h -- plain structs passed from the host launchers to the kernels.
#pragma once

#include <stdint.h>

namespace pa {

enum { KV_BF16 = 0, KV_FP8 = 1, KV_NVFP4 = 2 };

// Wait-site ids recorded in the error word when a bounded wait gives up.
enum {
  SITE_DEC_EMPTY = 101,
  SITE_DEC_FULL = 102,
  SITE_PRE_Q = 201,
  SITE_PRE_KV_EMPTY = 202,
  SITE_PRE_KV_FULL = 203,
  SITE_PRE_S_FULL = 204,
  SITE_PRE_S_FREE = 205,
  SITE_PRE_P_FULL = 206,
  SITE_PRE_O_DONE = 207,
  SITE_PRE_DEQ = 208,
  SITE_PRE_STG = 209,
  SITE_PRE_SF = 210,
  SITE_APPEND_POS = 301,  // append: more new tokens than the sequence holds, or a page id out of range
};

// Decode work list entry: one page-aligned chunk of one sequence.
struct DecodeChunk {
  int b;           // sequence
  int page_begin;  // first logical page (index into the sequence's page list)
  int page_end;    // one past the last logical page
  int split;       // index of this chunk among the sequence's chunks
};

struct DecodeParams {
  const uint16_t* q;  // bf16 [batch, Hq, d_qk]
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* kv_last_page_len;
  const float* k_scale;  // device scalar or nullptr (bf16)
  const float* v_scale;
  uint16_t* out;  // bf16 [batch, Hq, d_vo]
  float* lse;     // [batch, Hq] or nullptr
  // workspace
  int* err;           // error word
  int* hdr;           // [0] number of chunks, [1] chunk pages
  DecodeChunk* chunks;
  int2* seq_info;     // per sequence: {first chunk row, number of chunks}
  float* ws_o;        // [max_chunks][Hq][d_vo] unnormalised partial outputs
  float2* ws_ml;      // [max_chunks][Hq] {running max (log2 units), running sum}
  int batch, Hq, Hkv, group, page_size, window_left;
  int max_chunks, target_chunks, forced_chunk_pages;
  int min_chunk_pages;  // pages of about 4 MiB of K and V of one kv head
  int grid;             // CTAs of the decode kernel
  int box_rows;   // rows per TMA box: min(page_size, tile tokens), a power of two
  int box_shift;  // log2(box_rows)
  int swz;        // 7 when the K/V smem tiles are 128B-swizzled, 0 when not
  // 1: one item per (sequence, kv head) over its whole visible range, written directly
  // (no planner, no split, no merge: problems whose every item fits one CTA's round)
  int direct;
  float sm_scale;
};

// Prefill work item: one tile of query rows (positions x heads of one kv head).
struct PrefillItem {
  int b;
  int q_begin;  // first new-token index (within the sequence) of the tile
  int kvh;
  int cost;     // keys visited (for ordering)
  // split KV: this item covers KV tiles [kv_t0, kv_t1) of the tile's range and writes
  // its normalised output and lse to partial slot `slot`; slot -1: the whole range,
  // written to the output
  int kv_t0, kv_t1, slot;
};

// split KV: the partial slots [slot0, slot0 + parts) of one (tile, kv head), merged into
// its output rows
struct PrefillMerge {
  int b, q_begin, kvh, slot0, parts;
};

struct PrefillParams {
  const uint16_t* q;  // bf16 [total_q, Hq, d_qk]
  const int32_t* qo_indptr;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* kv_last_page_len;
  const float* k_scale;
  const float* v_scale;
  const uint8_t* kv_cache;  // for the plain-load (dequantising) producer
  const uint8_t* sf;
  uint16_t* out;  // bf16 [total_q, Hq, d_vo]
  float* lse;
  int* err;
  int* hdr;  // [0] number of items, [1] number of merges, [2] 1: items are per-tile records
  PrefillItem* items;
  int* tile_off;  // [batch + 1] first tile of each sequence
  // head_dim_vo 512: P tiles of the first pass ([128 rows][128 keys] bf16, in the MMA's
  // shared-memory image) and the softmax base of each row, per CTA, so that the second
  // pass reuses P instead of recomputing S; items with more than reuse_tiles KV tiles
  // recompute.
  uint8_t* p_scratch;   // [grid][reuse_tiles][32 KB]
  float* m_scratch;     // [grid][reuse_tiles][128]
  int reuse_tiles;
  int batch, total_q, Hq, Hkv, group, page_size, window_left, causal, num_pages;
  int rows_per_tile;  // query positions per 128-row tile (128 / group)
  int pair;           // 1: items span two tiles, computed by the two CTAs of a cluster
  // split KV (short queries over long KV): when split_target > 0 and the tiles x kv heads
  // are fewer than split_target, the planner splits long KV ranges into chunks so that
  // about 2 x split_target items exist; each chunk writes [128 rows][d_vo] fp32 and
  // [128] lse to its slot, merged afterwards (hdr[1] = number of merges)
  int split_target;
  float* part_o;
  float* part_lse;
  PrefillMerge* merges;
  int max_slots;
  // optional custom mask: bit mask_indptr[b] * 8 + i * kv_len + j (bit k of a byte is
  // its 2^k bit) lets new token i of sequence b attend key j; nullptr = none
  const uint8_t* mask;
  const int64_t* mask_indptr;
  int max_items;
  // rows one page occupies in the K/V tiles the kernel reads: page_size, or 8 for pages
  // of 1, 2 or 4 tokens read from a copy that pads every page to 8 rows (rows past the
  // page's tokens are zero); a 128-row KV tile then holds 128 / box_rows pages, i.e.
  // tile_tok = 128 / box_rows * page_size tokens
  int box_rows;
  int tile_tok;
  int out_v8;  // out is 32-byte aligned: the epilogue writes whole 32-byte sectors
  int swz;
  float sm_scale;
};

// Pages -> bf16 copy for the prefill (see prefill_dequant.cuh): FP8 / NVFP4 pages
// converted, and pages of fewer than 8 tokens (any dtype) padded to 8 rows per kv head
struct DequantParams {
  const uint8_t* cache;  // the caller's pages
  const uint8_t* sf;     // NVFP4 block-scale pool (same page indexing)
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  uint16_t* shadow;      // bf16 pages, same page index
  int batch, Hkv, page_size;
  int out_rows;          // rows per kv head in a copy page: page_size, or 8 when padding
};

// New tokens' K / V (bf16) -> the paged cache, converted to the cache's element type
// (see append.cu)
struct AppendParams {
  const uint16_t* k_new;  // bf16 [total_new, Hkv, d_qk]
  const uint16_t* v_new;  // bf16 [total_new, Hkv, d_vo]
  const int32_t* append_indptr;  // [batch + 1]
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* kv_last_page_len;
  const float* k_scale;  // FP8: per-tensor scale; NVFP4: global scale (device scalars)
  const float* v_scale;
  uint8_t* cache;        // pages in the cache's element type
  uint8_t* sf;           // NVFP4 block-scale pool (same page indexing)
  int* err;
  int batch, total_new, num_pages, Hkv, d_qk, d_vo, page_size;
};

}  // namespace pa

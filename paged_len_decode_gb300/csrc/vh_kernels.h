// vh_kernels.h -- parameter blocks and launchers shared by the host layer and
// the kernel translation units (internal; the public interface is vh.h).
#pragma once

#include <cstdint>
#include <cuda.h>  // CUtensorMap (the type only: the library does not link the driver library)
#include <cuda_runtime.h>

namespace vh {

// Per-step plan (vh_decode_plan): a header of 8 ints (kPlanMagic, B, N, T,
// n_eff, fused rules, max_pages_per_seq, P), the per-row arrays in the
// attention kernel's shared-memory layout (tile prefix sums cum[B+1], lengths
// [B], positions [B], each 16-byte aligned), and one record of kPlanRecInts
// ints per CTA: t0, t1, first row, last row, then the page ids of the range's
// first 64 tiles and, for 8-token pages, of the second page of each of them.
constexpr int kPlanMagic = 0x56485031;
constexpr int kPlanWindow = 64;
constexpr int kPlanRecInts = 4 + 2 * kPlanWindow;

struct RopeAppendParams {
  const uint16_t* q;
  const uint16_t* k_new;
  const uint16_t* v_new;
  const float* cos_sin;
  int max_pos;
  const int32_t* positions;
  uint16_t* k_cache;
  uint16_t* v_cache;
  long long page_stride;
  long long token_stride;
  long long head_stride;       // elements between the kv heads of one token slot
  int num_pages;
  const int32_t* page_table;
  int max_pages_per_seq;
  const int32_t* seq_lens;
  const int32_t* active;
  float* q_rot;
  int32_t* err_flag;
  const float* q_norm_w;       // [D] RMSNorm weights of q heads, or null
  const float* k_norm_w;       // [D] RMSNorm weights of the new k heads, or null
  float norm_eps;
  int rope_interleaved;        // RoPE pairs (2i, 2i+1) instead of (i, i + D/2)
  int f16;                     // 16-bit elements are fp16 (else bf16)
  int B, Hq, Hkv, D, P;
};

// Shared-memory plan of the attention kernel (byte offsets from the dynamic
// shared-memory base, rounded up to 1024 bytes) and the split plan parameters.
struct AttnParams {
  // K and V caches as 4-D tensors (head_dim, token, kv head, page) with the
  // 128-byte swizzle: boxes of 64 elements x 16 tokens x Hc heads for full
  // tiles (tmap_k, tmap_v), and of 64 x 8 tokens x 1 head (tmap_k8, tmap_v8)
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
  CUtensorMap tmap_k8;
  CUtensorMap tmap_v8;
  int tm_tok_dim;              // dimension of the token index in the 8-token maps (1 or 2; the head is the other)
  int full_boxes;              // 1: full tiles take the 16-token maps; 0: every tile takes 8-token boxes
  // attention over the cache (both kernels)
  const float* q_rot;          // [B][Hq][D] fp32 rotated q (three-call path)
  const uint16_t* k_cache;
  const uint16_t* v_cache;
  long long page_stride;
  long long token_stride;
  long long head_stride;       // elements between the kv heads of one token slot (D: heads contiguous)
  int num_pages;
  const int32_t* page_table;
  int max_pages_per_seq;
  const int32_t* seq_lens;
  const int32_t* active;
  uint16_t* out;
  float scale_log2;            // softmax scale * log2(e)
  int4* plan;                  // [B] split plan (three-call path)
  int* counters;               // [groups][B] pieces delivered per row (fused path; zero between calls)
  float* part_o;               // [groups][N][2][Hc*G][D]
  float* part_lse;             // [groups][N][2][Hc*G]   (base-2 log-sum-exp)
  int32_t* err_flag;
  // per-step plan written by vh_decode_plan (used when planned != 0)
  const int* plan_hdr;
  const int* plan_rows;        // copied as one block into the shared arrays at cum_off
  const int* plan_recs;
  int planned;
  int rows_bytes;              // bytes of the per-row arrays (cum | lens | pos)
  // fused step only: RoPE of q and k, append of the new token, in-kernel combine
  const uint16_t* q;           // [B][Hq][D] new queries (bf16 / fp16)
  const uint16_t* k_new;       // [B][Hkv][D]
  const uint16_t* v_new;       // [B][Hkv][D]
  const float* cos_sin;        // [max_pos][D]
  int max_pos;
  const int32_t* positions;    // [B] or null (seq_len - 1)
  uint16_t* k_cache_w;         // writable views of the cache for the append
  uint16_t* v_cache_w;
  const float* q_norm_w;       // [D] per-head RMSNorm weights before RoPE, or null
  const float* k_norm_w;
  float norm_eps;
  int rope_interleaved;        // RoPE pairs (2i, 2i+1) instead of (i, i + D/2)
  // element type of q, k_new, v_new, the cache and out: fp16 if set, else bf16
  int f16;
  // shapes and plan
  int B, Hq, Hkv, D, G, P;
  int Hc;                      // kv heads per CTA = consumer warps
  int groups;                  // Hkv / Hc (gridDim.y)
  int N;                       // CTAs per group (gridDim.x)
  int stages;
  int min_tiles;               // lower bound on tiles per CTA when the work list is short
  int prefetch_kv;             // fused: request the first stages of cached K/V before the dependency wait
  int early_q;                 // thread 0 requests the first segment's q rows right after the wait
  int host_io;                 // fused: q is host memory read in place (plain loads; the RoPE row is still copied)
  int l2_tiles;                // tiles after the first `stages` prefetched into L2 right after the wait
  int stage_bytes;             // K then V of one tile: [D/64][Hc][16 tokens][128 B swizzled] each
  int q_bytes;                 // bytes reserved for the q staging buffer
  int q_row_bytes;             // padded shared-memory stride of a staged q row
  int q_tx_bytes;              // bytes the q copies deliver
  int q_off, cum_off, len_off, pos_off, meta_off, bar_off;
  int qs_off;                  // per-warp fp32 q rows (rotated), padded: G * (D*4 + 32) bytes per warp
  int smem_bytes;
  int fused;
};

// The per-step plan kernel: the same work list the attention kernel would
// derive, written once for every attention launch of a decode step.
struct PlanParams {
  const int32_t* seq_lens;
  const int32_t* active;
  const int32_t* positions;    // fused rules only; null: seq_len - 1
  const int32_t* page_table;   // null: contiguous cache
  int max_pages_per_seq;
  int max_pos;
  int P, B, N, min_tiles;
  int fused;                   // fused rules: rows with a position outside [0, max_pos) get no tiles
  int* hdr;
  int* rows;                   // cum [B+1] | lens [B] at len_idx | pos [B] at pos_idx
  int* recs;
  int len_idx, pos_idx;
  int32_t* err_flag;
};

struct CombineParams {
  const int4* plan;
  const float* part_o;
  const float* part_lse;
  uint16_t* out;
  int B, Hq, D, Hc, G, N;
  int f16;
};

cudaError_t launch_rope_table(float* cos_sin, int max_pos, int D, double theta, cudaStream_t stream);
cudaError_t launch_wait_timeout_selftest(int32_t* err_flag, cudaStream_t stream);
cudaError_t launch_rope_kv_append(const RopeAppendParams& p, cudaStream_t stream);
cudaError_t prepare_decode_attn(int D, int G, int max_smem);  // once per device, every variant
cudaError_t launch_decode_attn(const AttnParams& p, cudaStream_t stream, bool pdl);
cudaError_t launch_decode_combine(const CombineParams& p, int groups, cudaStream_t stream);
cudaError_t prepare_decode_plan(int max_smem);  // once per device
cudaError_t launch_decode_plan(const PlanParams& p, cudaStream_t stream);
cudaError_t decode_attn_occupancy(const AttnParams& p, int* blocks_per_sm);

}  // namespace vh
